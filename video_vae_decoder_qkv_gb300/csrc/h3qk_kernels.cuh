// Device side of libh3qk: the fused QK-prep kernels for sm_103a.
//
// The path is bound by HBM bandwidth (about 12 bytes moved per Q/K/V element
// in 16-bit mode and ~15 flops per element), so there is no contraction and
// no tensor-core work here.  The design choices:
//  - one head row (D channels) is spread over LPR = next_pow2(D/8) lanes,
//    each lane owning 8 neighbouring channels = one 128-bit load or store;
//    a warp therefore covers 32/LPR consecutive token rows, so each warp-wide
//    store writes 32/LPR contiguous output rows of one head (512 B at D=128);
//  - the RMS reduction is a fixed tree: each lane sums its 8 squares left to
//    right, then xor-shuffles at offsets LPR/2 ... 1 (a halving tree whose
//    every lane ends holding the same sum);
//  - sin/cos of the rotary angles are computed once per token row in the
//    lanes that own the channels, and reused for every head and for both Q
//    and K (2H head rows per evaluation);
//  - the e4m3 cast is a read-only amax pass (lane max -> warp -> block -> one
//    atomicMax per tensor per block) followed by a cast pass that recomputes
//    the 16-bit values; two stream-ordered launches, no grid-wide wait.
//
// Every rounding point is an explicit correctly rounded intrinsic
// (__fmul_rn, __fadd_rn, __fsqrt_rn, __frcp_rn, __fmaf_rn), so compiler
// contraction flags cannot change a result bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace h3qk {

constexpr int kMaxPairs = 128;       // rotary_dim <= 256
constexpr int kWarpsPerBlock = 8;
constexpr int kThreads = 32 * kWarpsPerBlock;
// Tuning knobs (compile-time; the defaults are the measured best):
// H3QK_CH chunks of 8 channels per lane, H3QK_UNROLL head rows per batch,
// H3QK_PIPE prefetch of the next batch, H3QK_MIN_BLOCKS resident blocks per SM
// asked of the register allocator.
#ifndef H3QK_CH
#define H3QK_CH 1
#endif
#ifndef H3QK_UNROLL
#define H3QK_UNROLL 4
#endif
#ifndef H3QK_PIPE
#define H3QK_PIPE 0
#endif
#ifndef H3QK_MIN_BLOCKS
#define H3QK_MIN_BLOCKS 1
#endif
constexpr int kChunksPerLane = H3QK_CH;
constexpr int kUnroll = H3QK_UNROLL;
constexpr bool kPipe = H3QK_PIPE != 0;

enum Mode : int { kOut16 = 0, kAmax = 1, kCast = 2 };

// Everything a launch needs, passed as one __grid_constant__ parameter.
struct Params {
    const uint16_t* qkv;
    const float* wq;
    const float* wk;
    const int32_t* pos;
    void* out[3];
    float* out_scales;
    unsigned int* amax_words;    // 3 words: binary32 bits of the running amax
    const unsigned int* scale_words;  // cast mode: amax_words (dynamic) or the static table
    int64_t rows;                // B*S
    int64_t seq;                 // S
    int64_t valid_len;
    int64_t row_stride;          // elements
    int32_t heads;
    int32_t head_dim;
    int32_t rotary_dim;
    int32_t n_axes;
    int32_t chunks;              // D / 8
    int32_t dynamic;             // cast mode: 1 dynamic, 0 static
    float eps;
    float inv_d;                 // 1/D when D is a power of two, else 0
    float inv_freq[kMaxPairs];   // per rotary pair
    uint8_t axis[kMaxPairs];     // position axis of each rotary pair
};

// ---------------------------------------------------------------------------
// Sine and cosine of a binary32 angle: the library's own routine (Cody & Waite
// additive reduction by pi/2 split into three binary32 parts, each step one
// fused multiply-add; Taylor series of sin to r^11 and cos to r^12 in Horner
// form; quadrant by j mod 4).  Constants: 2/pi, pi/2 and its two tails, and
// +-1/n!, each rounded to binary32.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void sincos_h3(float a, float& s_out, float& c_out)
{
    constexpr float kTwoOverPi = 0x1.45f306p-1f;
    constexpr float kP1 = 0x1.921fb6p+0f;
    constexpr float kP2 = -0x1.777a5cp-25f;
    constexpr float kP3 = -0x1.ee59dap-50f;
    constexpr float kS3 = -0x1.555556p-3f, kS5 = 0x1.111112p-7f, kS7 = -0x1.a01a02p-13f;
    constexpr float kS9 = 0x1.71de3ap-19f, kS11 = -0x1.ae6456p-26f;
    constexpr float kC2 = -0x1.000000p-1f, kC4 = 0x1.555556p-5f, kC6 = -0x1.6c16c2p-10f;
    constexpr float kC8 = 0x1.a01a02p-16f, kC10 = -0x1.27e4fcp-22f, kC12 = 0x1.1eed8ep-29f;

    const float j = rintf(__fmul_rn(a, kTwoOverPi));
    float r = __fmaf_rn(-j, kP1, a);
    r = __fmaf_rn(-j, kP2, r);
    r = __fmaf_rn(-j, kP3, r);
    const float r2 = __fmul_rn(r, r);
    float ps = __fmaf_rn(kS11, r2, kS9);
    ps = __fmaf_rn(ps, r2, kS7);
    ps = __fmaf_rn(ps, r2, kS5);
    ps = __fmaf_rn(ps, r2, kS3);
    const float sr = __fmaf_rn(ps, __fmul_rn(r2, r), r);
    float pc = __fmaf_rn(kC12, r2, kC10);
    pc = __fmaf_rn(pc, r2, kC8);
    pc = __fmaf_rn(pc, r2, kC6);
    pc = __fmaf_rn(pc, r2, kC4);
    pc = __fmaf_rn(pc, r2, kC2);
    const float cr = __fmaf_rn(pc, r2, 1.0f);
    const int q = static_cast<int>(j) & 3;
    float s, c;
    if (q == 0) { s = sr; c = cr; }
    else if (q == 1) { s = cr; c = -sr; }
    else if (q == 2) { s = -sr; c = -cr; }
    else { s = -cr; c = sr; }
    s_out = s;
    c_out = c;
}

// ---------------------------------------------------------------------------
// 16-bit formats.
// ---------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ float2 widen2(uint32_t w)
{
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    }
}

// Round two binary32 values to the 16-bit type (nearest even), lo in the low half.
template <bool BF16>
__device__ __forceinline__ uint32_t round2(float lo, float hi)
{
    if constexpr (BF16) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&b);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// Two e4m3 codes (round to nearest even, saturating at +-448), lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 load16(const uint16_t* p)
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------------------
// The kernel.  A head row's C = D/8 chunks (8 channels = 16 bytes each) sit
// on LPR lanes, CH chunks per lane (chunks c, c+LPR, ..., LPR*CH =
// next_pow2(C)); a warp covers TPW = 32/LPR token rows.  Each warp walks
// groups of TPW rows (grid-stride) and, for each, the 3*H head rows
// Q[0..H), K[0..H), V[0..H) in batches of U, optionally loading the next
// batch before computing the current one (PIPE).  The reduction tree is the
// same for every (LPR, CH): the first log2(CH) halving levels pair chunks
// held by the same lane, the rest are xor shuffles.
// MODE kOut16 writes 16-bit head-major outputs; kAmax reduces max |y| per
// tensor; kCast writes e4m3 codes under the dynamic or static factors.
// ---------------------------------------------------------------------------
template <int CH, int U>
struct Batch {
    uint4 v[U][CH];
};

template <int LPR, int CH, int U>
__device__ __forceinline__ void load_batch(Batch<CH, U>& bt, const uint16_t* row, int j0, int H,
                                           int D, int64_t HD, const bool (&act)[CH])
{
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int j = j0 + u;
        const int part = j / H;
        const int h = j - part * H;
        const bool in = j < 3 * H;
#pragma unroll
        for (int q = 0; q < CH; ++q) {
            bt.v[u][q] = make_uint4(0u, 0u, 0u, 0u);
            if (in && act[q]) bt.v[u][q] = load16(row + part * HD + static_cast<int64_t>(h) * D + 8 * q * LPR);
        }
    }
}

template <bool BF16, int LPR, int CH, int U, bool PIPE, int MODE>
__global__ void __launch_bounds__(kThreads, H3QK_MIN_BLOCKS) qkprep_kernel(const __grid_constant__ Params p)
{
    constexpr int TPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    const int c = lane % LPR;
    bool chunk_on[CH];
#pragma unroll
    for (int q = 0; q < CH; ++q) chunk_on[q] = c + q * LPR < p.chunks;
    const int H = p.heads;
    const int D = p.head_dim;
    const int64_t HD = static_cast<int64_t>(H) * D;
    const int64_t head_stride = p.seq * D;  // between heads of one output tensor
    const int64_t n_groups = (p.rows + TPW - 1) / TPW;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

    // Cast factors (each thread derives them; block 0 publishes the descales).
    float fac[3] = {1.0f, 1.0f, 1.0f};
    if constexpr (MODE == kCast) {
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            // One load from whichever table this mode uses (never a NULL pointer).
            const float a = __uint_as_float(__ldcg(p.scale_words + t));
            const bool ok = a >= 1.17549435e-38f && a <= 3.40282347e+38f;
            float s = 1.0f, f = 1.0f;
            if (ok) {
                if (p.dynamic) {
                    s = __fdiv_rn(a, 448.0f);
                    f = __fdiv_rn(448.0f, a);
                } else {
                    s = a;
                    f = __frcp_rn(a);
                }
            }
            fac[t] = f;
            if (blockIdx.x == 0 && threadIdx.x == 0) p.out_scales[t] = s;
        }
    }

    // This lane's norm weights of Q and K, 8 per chunk.
    float wq[CH][8], wk[CH][8];
#pragma unroll
    for (int q = 0; q < CH; ++q) {
        if (chunk_on[q]) {
            const float4* q4 = reinterpret_cast<const float4*>(p.wq + 8 * (c + q * LPR));
            const float4* k4 = reinterpret_cast<const float4*>(p.wk + 8 * (c + q * LPR));
            const float4 a = __ldg(q4), b = __ldg(q4 + 1), e = __ldg(k4), f = __ldg(k4 + 1);
            wq[q][0] = a.x; wq[q][1] = a.y; wq[q][2] = a.z; wq[q][3] = a.w;
            wq[q][4] = b.x; wq[q][5] = b.y; wq[q][6] = b.z; wq[q][7] = b.w;
            wk[q][0] = e.x; wk[q][1] = e.y; wk[q][2] = e.z; wk[q][3] = e.w;
            wk[q][4] = f.x; wk[q][5] = f.y; wk[q][6] = f.z; wk[q][7] = f.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) wq[q][k] = wk[q][k] = 0.0f;
        }
    }

    float amax[3] = {0.0f, 0.0f, 0.0f};

    for (int64_t g = warp0; g < n_groups; g += n_warps) {
        const int64_t r = g * TPW + sub;
        int64_t b = 0, s = 0;
        bool act_row = false;
        if (r < p.rows) {
            b = r / p.seq;
            s = r - b * p.seq;
            act_row = s < p.valid_len;
        }
        bool act[CH];
#pragma unroll
        for (int q = 0; q < CH; ++q) act[q] = act_row && chunk_on[q];

        // Rotary cos/sin of this lane's pairs (pair index 4*(c + q*LPR) + k).
        float cs[CH][4], sn[CH][4];
        bool rot[CH][4];
#pragma unroll
        for (int q = 0; q < CH; ++q)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int pair = 4 * (c + q * LPR) + k;
                rot[q][k] = 2 * pair < p.rotary_dim;
                cs[q][k] = 1.0f;
                sn[q][k] = 0.0f;
                if (rot[q][k] && act[q]) {
                    const float pv = static_cast<float>(__ldg(p.pos + r * p.n_axes + p.axis[pair]));
                    sincos_h3(__fmul_rn(pv, p.inv_freq[pair]), sn[q][k], cs[q][k]);
                }
            }

        const uint16_t* row = p.qkv + r * p.row_stride + 8 * c;
        const int64_t obase = (b * H * p.seq + s) * D + 8 * c;

        Batch<CH, U> cur;
        if constexpr (PIPE) load_batch<LPR, CH, U>(cur, row, 0, H, D, HD, act);
        for (int j0 = 0; j0 < 3 * H; j0 += U) {
            Batch<CH, U> nxt;
            if constexpr (PIPE) {
                if (j0 + U < 3 * H) load_batch<LPR, CH, U>(nxt, row, j0 + U, H, D, HD, act);
            } else {
                load_batch<LPR, CH, U>(cur, row, j0, H, D, HD, act);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u;
                if (j >= 3 * H) break;                 // warp-uniform
                const int part = j / H;
                const int h = j - part * H;
                uint32_t y[CH][4];
                if (part < 2) {
                    float x[CH][8];
                    float acc[CH];
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        const uint32_t wv[4] = {cur.v[u][q].x, cur.v[u][q].y, cur.v[u][q].z, cur.v[u][q].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 f = widen2<BF16>(wv[k]);
                            x[q][2 * k] = f.x;
                            x[q][2 * k + 1] = f.y;
                        }
                        // Sum of squares of one chunk: 8 channels left to right.
                        acc[q] = __fmul_rn(x[q][0], x[q][0]);
#pragma unroll
                        for (int k = 1; k < 8; ++k) acc[q] = __fadd_rn(acc[q], __fmul_rn(x[q][k], x[q][k]));
                    }
                    // Halving tree: levels pairing chunks of this lane, then shuffles.
#pragma unroll
                    for (int o = CH / 2; o >= 1; o >>= 1)
#pragma unroll
                        for (int q = 0; q < o; ++q) acc[q] = __fadd_rn(acc[q], acc[q + o]);
                    float ss = acc[0];
#pragma unroll
                    for (int o = LPR / 2; o >= 1; o >>= 1)
                        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
                    const float ms = p.inv_d != 0.0f ? __fmul_rn(ss, p.inv_d)
                                                     : __fdiv_rn(ss, static_cast<float>(D));
                    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
#pragma unroll
                    for (int q = 0; q < CH; ++q)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float w0 = part == 0 ? wq[q][2 * k] : wk[q][2 * k];
                            const float w1 = part == 0 ? wq[q][2 * k + 1] : wk[q][2 * k + 1];
                            const float a0 = __fmul_rn(__fmul_rn(x[q][2 * k], inv), w0);
                            const float a1 = __fmul_rn(__fmul_rn(x[q][2 * k + 1], inv), w1);
                            uint32_t n2 = round2<BF16>(a0, a1);
                            if (rot[q][k]) {
                                const float2 uv = widen2<BF16>(n2);
                                const float ro = __fsub_rn(__fmul_rn(uv.x, cs[q][k]), __fmul_rn(uv.y, sn[q][k]));
                                const float rv = __fadd_rn(__fmul_rn(uv.x, sn[q][k]), __fmul_rn(uv.y, cs[q][k]));
                                n2 = round2<BF16>(ro, rv);
                            }
                            y[q][k] = n2;
                        }
                } else {
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        y[q][0] = cur.v[u][q].x;
                        y[q][1] = cur.v[u][q].y;
                        y[q][2] = cur.v[u][q].z;
                        y[q][3] = cur.v[u][q].w;
                    }
                }

#pragma unroll
                for (int q = 0; q < CH; ++q) {
                    if (!act[q]) continue;
                    const int64_t off = obase + h * head_stride + 8 * q * LPR;
                    if constexpr (MODE == kOut16) {
                        uint16_t* dst = static_cast<uint16_t*>(p.out[part]) + off;
                        *reinterpret_cast<uint4*>(dst) = make_uint4(y[q][0], y[q][1], y[q][2], y[q][3]);
                    } else if constexpr (MODE == kAmax) {
                        float m = 0.0f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 f = widen2<BF16>(y[q][k]);
                            m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
                        }
                        if (part == 0) amax[0] = fmaxf(amax[0], m);
                        else if (part == 1) amax[1] = fmaxf(amax[1], m);
                        else amax[2] = fmaxf(amax[2], m);
                    } else {
                        const float fa = part == 0 ? fac[0] : (part == 1 ? fac[1] : fac[2]);
                        uint32_t cw[2];
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const float2 f0 = widen2<BF16>(y[q][2 * k]);
                            const float2 f1 = widen2<BF16>(y[q][2 * k + 1]);
                            cw[k] = e4m3x2(__fmul_rn(f0.x, fa), __fmul_rn(f0.y, fa)) |
                                    (e4m3x2(__fmul_rn(f1.x, fa), __fmul_rn(f1.y, fa)) << 16);
                        }
                        uint8_t* dst = static_cast<uint8_t*>(p.out[part]) + off;
                        *reinterpret_cast<uint2*>(dst) = make_uint2(cw[0], cw[1]);
                    }
                }
            }
            if constexpr (PIPE) cur = nxt;
        }
    }

    if constexpr (MODE == kAmax) {
        __shared__ float red[3][kWarpsPerBlock];
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            float m = amax[t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) red[t][threadIdx.x >> 5] = m;
        }
        __syncthreads();
        if (threadIdx.x < 3) {
            float m = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarpsPerBlock; ++w) m = fmaxf(m, red[threadIdx.x][w]);
            // Non-negative binary32 values order like their bit patterns.
            if (m > 0.0f) atomicMax(p.amax_words + threadIdx.x, __float_as_uint(m));
        }
    }
}

// Zero the three amax words of a dynamic call.
__global__ void amax_init_kernel(unsigned int* words)
{
    if (threadIdx.x < 3) words[threadIdx.x] = 0u;
}

}  // namespace h3qk
