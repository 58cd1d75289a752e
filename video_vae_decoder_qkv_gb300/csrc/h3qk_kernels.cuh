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
#include <type_traits>

namespace h3qk {

constexpr int kMaxPairs = 128;       // rotary_dim <= 256
constexpr int kWarpsPerBlock = 8;    // head_dim > 64; see Shape for head_dim <= 64
// Tuning knobs (compile-time; the defaults are the measured best):
// H3QK_CH_<MODE> chunks of 8 channels per lane (1, 2 or 4; default H3QK_CH),
// and per mode a five-digit code "U UV MIN_BLOCKS PF S": Q/K head rows per batch of
// loads, V head rows per batch, resident blocks per SM asked of the register
// allocator, the L2 bulk prefetch distance in batches (0 = off), and the
// depth of the per-warp shared-memory pipeline (0 = loads straight into
// registers; S > 0: S stages of cp.async copies, V batches of U rows).
#ifndef H3QK_CH
#define H3QK_CH 2
#endif
#ifndef H3QK_CH_OUT16
#define H3QK_CH_OUT16 H3QK_CH
#endif
#ifndef H3QK_CH_AMAX
#define H3QK_CH_AMAX H3QK_CH
#endif
#ifndef H3QK_CH_CAST
#define H3QK_CH_CAST H3QK_CH
#endif
#ifndef H3QK_CH_SAGE
#define H3QK_CH_SAGE H3QK_CH
#endif

#ifndef H3QK_TUNE_OUT16
#define H3QK_TUNE_OUT16 44202
#endif
#ifndef H3QK_TUNE_AMAX
#define H3QK_TUNE_AMAX 24303
#endif
#ifndef H3QK_TUNE_CAST
#define H3QK_TUNE_CAST 24303
#endif
#ifndef H3QK_TUNE_SAGE
#define H3QK_TUNE_SAGE 44204
#endif

// kRotFirst instances (see RotMode) are used from this many lanes per head
// row up; narrower heads take the general instance (at head_dim 64 the
// kRotFirst cast spills and measured 10 % slower).
#ifndef H3QK_ROT_FIRST_MIN_LPR
#define H3QK_ROT_FIRST_MIN_LPR 8
#endif

// 1: the kRotFirst cast instances keep the rotary cos/sin of a row group in
// shared memory instead of registers (see kAngSmem in the kernel).
#ifndef H3QK_SMEM_ANGLES
#define H3QK_SMEM_ANGLES 1
#endif

// Head split of the amax pass: its warps take 32/LPR/H head rows of H
// interleaved head batches each (see HS in the kernel); 1 = one head batch
// of 32/LPR token rows, as every other mode.
#ifndef H3QK_AMAX_HEAD_SPLIT
#define H3QK_AMAX_HEAD_SPLIT 1
#endif

// 1: the amax pass walks each work item backwards (see kBack in the kernel).
#ifndef H3QK_AMAX_BACK
#define H3QK_AMAX_BACK 1
#endif

// The amax pass's pairwise second bound (qk_pair_may_exceed) runs in the
// instances whose warps hold at least this many token rows.
#ifndef H3QK_AMAX_PAIR_MIN_TPW
#define H3QK_AMAX_PAIR_MIN_TPW 1
#endif

// kCastCount is the cast that also counts clipped values (opts.sat_counts):
// a separate instance, so that the plain cast carries no counter state.
enum Mode : int { kOut16 = 0, kAmax = 1, kCast = 2, kSage = 3, kCastCount = 4 };

template <int CODE, int CH_>
struct TuneT {
    static constexpr int CH = CH_;               // chunks of 8 channels per lane
    static constexpr int U = CODE / 10000;       // Q/K head rows per batch of loads
    static constexpr int UV = CODE / 1000 % 10;  // V head rows per batch (register path)
    static constexpr int MB = CODE / 100 % 10;   // __launch_bounds__ minimum blocks per SM
    static constexpr int PF = CODE / 10 % 10;    // L2 prefetch distance in batches
    static constexpr int S = CODE % 10;          // shared-memory pipeline stages (0 = none)
    static_assert(U >= 1 && UV >= 1 && MB >= 1, "tuning code digits U, UV, MIN_BLOCKS must be >= 1");
};
template <int MODE> struct Tune;
template <> struct Tune<kOut16> : TuneT<H3QK_TUNE_OUT16, H3QK_CH_OUT16> {};
template <> struct Tune<kAmax> : TuneT<H3QK_TUNE_AMAX, H3QK_CH_AMAX> {};
template <> struct Tune<kCast> : TuneT<H3QK_TUNE_CAST, H3QK_CH_CAST> {};
template <> struct Tune<kSage> : TuneT<H3QK_TUNE_SAGE, H3QK_CH_SAGE> {};
template <> struct Tune<kCastCount> : TuneT<H3QK_TUNE_CAST, H3QK_CH_CAST> {};

// Tuning codes of the instances whose warps hold 8 or more token rows (LPR <=
// 4, head_dim <= 64), same digits; their MIN_BLOCKS digit is unused (Shape
// below sets it).  The 16-bit pass takes batches of 2 rows and 3 stages
// there (4 % faster than 4 rows and 2 stages at this block shape).
#ifndef H3QK_SMALL_TUNE_OUT16
#define H3QK_SMALL_TUNE_OUT16 24203
#endif
#ifndef H3QK_SMALL_TUNE_AMAX
#define H3QK_SMALL_TUNE_AMAX H3QK_TUNE_AMAX
#endif
#ifndef H3QK_SMALL_TUNE_CAST
#define H3QK_SMALL_TUNE_CAST H3QK_TUNE_CAST
#endif
#ifndef H3QK_SMALL_TUNE_SAGE
#define H3QK_SMALL_TUNE_SAGE H3QK_TUNE_SAGE
#endif
template <int MODE>
constexpr int small_tune_code()
{
    return MODE == kOut16 ? H3QK_SMALL_TUNE_OUT16
                          : (MODE == kAmax ? H3QK_SMALL_TUNE_AMAX
                                           : (MODE == kCast || MODE == kCastCount ? H3QK_SMALL_TUNE_CAST
                                                                                  : H3QK_SMALL_TUNE_SAGE));
}
// The tuning an instance uses: its mode's, or the small-head code above.
template <int MODE, int LPR>
using TuneL = typename std::conditional<(LPR <= 4), TuneT<small_tune_code<MODE>(), Tune<MODE>::CH>, Tune<MODE>>::type;

// Block shape of the instances whose warps hold 8 or more token rows (LPR <= 4,
// head_dim <= 64), per mode as a code "W MB": warps per block (1 or 2 digits)
// and the resident blocks per SM asked of the register allocator.  Their
// per-row work (the reduction, the root and reciprocal, the angles) weighs
// twice as much per byte as at head_dim 128.  Measured best: 16-bit output
// in blocks of 10 warps, 2 per SM (20 warps of up to 96 registers, against
// 8 x 2); amax and cast in blocks of 5 warps, 4 per SM (20 warps of up to 96
// registers, against 24 warps of 80 that spill); the sage outputs in blocks
// of 4 warps with registers for 4 per SM (its four-stage pipeline takes
// 64 KB per block, so 3 reside: 12 warps).  The larger heads keep
// 8 warps per block and the MIN_BLOCKS digit of their tuning code.
#ifndef H3QK_SMALL_OUT16
#define H3QK_SMALL_OUT16 102
#endif
#ifndef H3QK_SMALL_AMAX
#define H3QK_SMALL_AMAX 54
#endif
#ifndef H3QK_SMALL_CAST
#define H3QK_SMALL_CAST 54
#endif
#ifndef H3QK_SMALL_SAGE
#define H3QK_SMALL_SAGE 44
#endif
template <int MODE>
constexpr int small_code()
{
    return MODE == kOut16 ? H3QK_SMALL_OUT16
                          : (MODE == kAmax ? H3QK_SMALL_AMAX
                                           : (MODE == kCast || MODE == kCastCount ? H3QK_SMALL_CAST : H3QK_SMALL_SAGE));
}
template <int MODE, int LPR>
struct Shape {
    static constexpr bool kSmall = LPR <= 4;
    static constexpr int W = kSmall ? small_code<MODE>() / 10 : kWarpsPerBlock;  // warps per block
    static constexpr int MB = kSmall ? small_code<MODE>() % 10 : Tune<MODE>::MB;  // blocks per SM
    static constexpr int NT = 32 * W;                                          // threads per block
    static_assert(W >= 1 && W <= 32 && MB >= 1, "block shape code: warps 1..32, blocks per SM >= 1");
};

// Dynamic shared memory of one block of an instance: S stages x U head rows x
// CH chunks x 32 lanes x 16 bytes per warp.
template <int LPR, int CH, int MODE>
constexpr size_t stage_bytes()
{
    return static_cast<size_t>(Shape<MODE, LPR>::W) * TuneL<MODE, LPR>::S * TuneL<MODE, LPR>::U * CH * 32 * 16;
}

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
    int64_t in_part_off[3];      // element offset of Q, K, V within an input row
    int64_t out_bstride;         // output element strides of item, token, head
    int64_t out_sstride;
    int64_t out_hstride;
    int32_t qk_first, qk_end;    // parts [qk_first, qk_end) of {Q=0, K=1} get norm + RoPE
    int32_t has_v;               // part 2 (V) is copied / cast
    int32_t slot[3];             // amax / scale / count slot of each part, -1 if unused
    const int32_t* valid_lens;   // per-item valid lengths (device), or null
    unsigned int* sat_counts;    // kCastCount: clipped-element counters (device); null otherwise
    float kv_scale;              // sage mode: factor of K (binary32 out) and V (binary16 out)
    int32_t chained;             // host only: launched as a programmatic dependent of the
                                 // call's previous kernel (see the griddepcontrol notes)
    int32_t reverse;             // walk the row groups from the last one down (the cast
                                 // after an amax pass: see the note in the kernel)
    unsigned int* dbg_status;    // debug builds: the check status words (see dbg_ok); else null
    int64_t dbg_out_elems;       // debug builds: elements of each output tensor the checks allow
    float2 one2;                 // {1, 1} and {-1, -1}: the unit factors of the packed sums
    float2 mone2;                // (see fma2 below); read at run time, never constants
    int64_t pf_span;             // elements of an input row the call reads ([0, pf_span))
    int32_t hs_shift;            // sliced launches: log2 of the head slices per row group
    int32_t hs_heads;            // sliced launches: heads per slice
    float inv_freq[kMaxPairs];   // per rotary pair
    uint8_t axis[kMaxPairs];     // position axis of each rotary pair
};

// ---------------------------------------------------------------------------
// Debug builds (H3QK_DEBUG_CHECKS=1): every global access of qkprep_kernel is
// checked against the extent of its buffer before it is made.  A failed check
// ORs its bit into status word 0, counts itself in word 1, keeps the first
// offending offset + 1 in words 2-3 (64-bit), and the access is skipped, so
// a wrong index is reported and never made.  Release builds compile every
// check to `true`.
// ---------------------------------------------------------------------------
#ifndef H3QK_DEBUG_CHECKS
#define H3QK_DEBUG_CHECKS 0
#endif
enum DbgCheck : unsigned int {
    kDbgInput = 1u,      // a 16-byte load of the packed rows
    kDbgOutput = 2u,     // a store of 8 output elements
    kDbgPositions = 4u,  // a position load
    kDbgLengths = 8u,    // a per-item valid length load
    kDbgSlot = 16u       // an amax word, descale or counter index
};
__device__ __forceinline__ bool dbg_ok(const Params& p, bool ok, unsigned int what, int64_t at)
{
    if constexpr (H3QK_DEBUG_CHECKS) {
        if (!ok && p.dbg_status) {
            atomicOr(p.dbg_status, what);
            atomicAdd(p.dbg_status + 1, 1u);
            atomicCAS(reinterpret_cast<unsigned long long*>(p.dbg_status + 2), 0ull,
                      static_cast<unsigned long long>(at) + 1ull);
        }
        return ok;
    } else {
        return true;
    }
}
// The checks of one access kind, by offset in elements of the buffer.
__device__ __forceinline__ bool dbg_in(const Params& p, int64_t at)
{
    return dbg_ok(p, at >= 0 && at + 8 <= (p.rows - 1) * p.row_stride + p.pf_span, kDbgInput, at);
}
__device__ __forceinline__ bool dbg_out(const Params& p, int64_t at)
{
    return dbg_ok(p, at >= 0 && at + 8 <= p.dbg_out_elems, kDbgOutput, at);
}
__device__ __forceinline__ bool dbg_slot(const Params& p, int slot)
{
    return dbg_ok(p, slot >= 0 && slot < 3, kDbgSlot, slot);
}

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

// Prefetch `bytes` bytes at p (16-byte aligned, a multiple of 16, inside the
// input) into L2 with one bulk request; no completion is awaited.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// One 16-byte asynchronous copy global -> shared (L2 only, no L1 allocation),
// and the commit / wait of the calling thread's copy groups.  A thread reads
// back only what it copied itself, so no barrier is involved.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Packed product: two binary32 multiplies in one instruction, each rounded to
// nearest even.  Used only where the product feeds no addition (the norm,
// the weight and the e4m3 factor): a packed product that feeds a packed add
// may be fused into a multiply-add by the code generator even with .rn and
// --fmad=false, which would drop a rounding.  Products that feed additions
// use __fmul_rn, which is never merged into a multiply-add.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Packed fused multiply-add, RN(a*b + c) per half.  With b = {1, 1} or
// {-1, -1} (run-time values from the parameter block, which the code
// generator cannot fold) it is a correctly rounded sum RN(c +- a) of an
// already rounded product a: the code generator cannot merge the product
// that feeds it into a multiply-add, because that product is the
// multiplicand here, not an addend.  So a packed product followed by this
// sum keeps both rounding points of the plain definition.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Packed sum RN(a + b) per half, for operands that are not fresh products
// (sums of the reduction tree).
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// A binary32 value rounded to the 16-bit type (nearest even), returned as
// binary32.  bfloat16: one conversion that packs the rounded value above a
// zero half, which is that value's binary32 bit pattern.
template <bool BF16>
__device__ __forceinline__ float round16f(float a)
{
    if constexpr (BF16) {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(a), "f"(0.0f));
        return __uint_as_float(d);
    } else {
        return __half2float(__float2half_rn(a));
    }
}
template <bool BF16>
__device__ __forceinline__ float2 round16f2(float2 v)
{
    if constexpr (BF16) {
        return make_float2(round16f<true>(v.x), round16f<true>(v.y));
    } else {
        __half2 h = __floats2half2_rn(v.x, v.y);
        return __half22float2(h);
    }
}

template <bool BF16>
__device__ __forceinline__ float hmax2_to_float(uint32_t m)
{
    const float2 f = widen2<BF16>(m);
    return fmaxf(f.x, f.y);
}

// Running max of packed 16-bit magnitudes in one instruction: each half of
// the result has magnitude max(|m|, |y|), NaN ignored (the other operand is
// kept), and the xor of the two sign bits as its sign.  Read it through
// hmax2x_to_float, which drops the signs.
template <bool BF16>
__device__ __forceinline__ uint32_t hmax2x(uint32_t m, uint32_t y)
{
    uint32_t r;
    if constexpr (BF16) {
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(y));
    } else {
        asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(y));
    }
    return r;
}

template <bool BF16>
__device__ __forceinline__ float hmax2x_to_float(uint32_t m)
{
    return hmax2_to_float<BF16>(m & 0x7fff7fffu);
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------
// One Q or K head row as seen by one lane: its CH chunks of 8 channels in
// `raw` (chunk q of lane c is chunk c + q*LPR of the row), the lane's weights
// `w` (CH*8 floats, chunk by chunk), the rotary cos/sin and flags of its 4
// pairs per chunk.  Computes the sum of squares (each chunk left to right;
// the halving tree's levels that pair chunks of this lane, then xor shuffles
// over LPR lanes), 1/sqrt(ss/D + eps), the weighted 16-bit norm and the
// rotation, and returns the 16-bit words.
// ---------------------------------------------------------------------------
template <bool BF16, int LPR, int CH>
__device__ __forceinline__ float qk_inv(const uint4 (&raw)[CH], float inv_d, float eps, int D, float (&x)[CH][8])
{
#pragma unroll
    for (int q = 0; q < CH; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = widen2<BF16>(word(raw[q], i));
            x[q][2 * i] = f.x;
            x[q][2 * i + 1] = f.y;
        }
    // Sum of squares of each chunk, channels left to right.
    float acc[CH];
#pragma unroll
    for (int q = 0; q < CH; ++q) {
        acc[q] = __fmul_rn(x[q][0], x[q][0]);
#pragma unroll
        for (int k = 1; k < 8; ++k) acc[q] = __fadd_rn(acc[q], __fmul_rn(x[q][k], x[q][k]));
    }
    // Halving tree: chunk c+q*LPR pairs with chunk c+(q+o)*LPR in this lane
    // for o = CH/2 ... 1, then xor shuffles over the LPR lanes.
#pragma unroll
    for (int o = CH / 2; o >= 1; o >>= 1)
#pragma unroll
        for (int q = 0; q < o; ++q) acc[q] = __fadd_rn(acc[q], acc[q + o]);
    float ss = acc[0];
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float ms = inv_d != 0.0f ? __fmul_rn(ss, inv_d) : __fdiv_rn(ss, static_cast<float>(D));
    return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

template <bool BF16, int LPR, int CH>
__device__ __forceinline__ void qk_row(const uint4 (&raw)[CH], const float4* w, const float (&cs)[CH][4],
                                       const float (&sn)[CH][4], const bool (&rot)[CH][4], float inv_d,
                                       float eps, int D, uint32_t (&y)[CH][4])
{
    float x[CH][8];
    const float inv = qk_inv<BF16, LPR, CH>(raw, inv_d, eps, D, x);
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int q = 0; q < CH; ++q) {
        const float4 wa = w[2 * q], wb = w[2 * q + 1];
        const float wq[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = mul2(mul2(make_float2(x[q][2 * i], x[q][2 * i + 1]), inv2),
                                  make_float2(wq[2 * i], wq[2 * i + 1]));
            const uint32_t n = round2<BF16>(a.x, a.y);
            const float2 uv = widen2<BF16>(n);
            const float ro = __fsub_rn(__fmul_rn(uv.x, cs[q][i]), __fmul_rn(uv.y, sn[q][i]));  // u c - v s
            const float rv = __fadd_rn(__fmul_rn(uv.x, sn[q][i]), __fmul_rn(uv.y, cs[q][i]));  // u s + v c
            y[q][i] = rot[q][i] ? round2<BF16>(ro, rv) : n;
        }
    }
}

// The same head row for the e4m3 modes, computed on packed pairs.  Pair p
// holds the lane's chunks 2p and 2p+1 (chunks c + 2p*LPR and c + (2p+1)*LPR
// of the row) side by side, element k of each, so every packed operation
// does the work of two chunks: the squares and their running sums (a packed
// product, then the unit-factor sum of fma2), the in-lane level of the
// halving tree, the two products of the norm, the 16-bit rounding and the
// rotation (four packed products and two unit-factor sums per two pairs of
// channels).  The rounding points are those of qk_row, one for one.
// w2 points at the lane's weights in pair layout: float2 {w(chunk 2p, k),
// w(chunk 2p+1, k)} at [p*8 + k].  cs2/sn2 hold the pairs' cos/sin in the
// same layout.  For each pair p and rotary pair slot i, sink(p, i, yu, yv)
// receives the results, already rounded to 16 bits and held as binary32:
// yu = channel 2i, yv = channel 2i+1 of chunks 2p (.x) and 2p+1 (.y).
// RM says which channels the rotation applies to (the same for every lane
// of a call, so the caller picks it once): kRotAll, every channel (no
// per-value choice); kRotFirst (two chunks per lane), every channel of the
// lane's first chunk and, when rot1 is set, all of its second chunk (one
// choice per value of the second chunk); kRotAny, per pair as rot says.
enum RotMode : int { kRotAny = 0, kRotAll = 1, kRotFirst = 2 };
template <bool BF16, int LPR, int CH, int RM, class Sink>
__device__ __forceinline__ void qk_row_pairs(const uint4 (&raw)[CH], const float2* w2, const float2 (&cs2)[CH / 2][4],
                                             const float2 (&sn2)[CH / 2][4], const bool (&rot)[CH][4], bool rot1,
                                             float inv_d, float eps, int D, float2 one2, float2 mone2, Sink&& sink)
{
    static_assert(RM != kRotFirst || CH == 2, "kRotFirst: two chunks per lane");
    static_assert(CH == 2 || CH == 4, "pairs of chunks");
    constexpr int NP = CH / 2;
    float2 X[NP][8];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = widen2<BF16>(word(raw[2 * p], i));
            const float2 b = widen2<BF16>(word(raw[2 * p + 1], i));
            X[p][2 * i] = make_float2(a.x, b.x);
            X[p][2 * i + 1] = make_float2(a.y, b.y);
        }
    // Sum of squares of each chunk, channels left to right (two chunks per pair).
    float2 A[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        A[p] = mul2(X[p][0], X[p][0]);
#pragma unroll
        for (int k = 1; k < 8; ++k) A[p] = fma2(mul2(X[p][k], X[p][k]), one2, A[p]);
    }
    // In-lane levels of the halving tree: chunk q pairs with chunk q + CH/2.
    if constexpr (NP == 2) A[0] = add2(A[0], A[1]);
    float ss = __fadd_rn(A[0].x, A[0].y);
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float ms = inv_d != 0.0f ? __fmul_rn(ss, inv_d) : __fdiv_rn(ss, static_cast<float>(D));
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 wp = reinterpret_cast<const float4*>(w2)[p * 4 + i];
            const float2 u = round16f2<BF16>(mul2(mul2(X[p][2 * i], inv2), make_float2(wp.x, wp.y)));
            const float2 v = round16f2<BF16>(mul2(mul2(X[p][2 * i + 1], inv2), make_float2(wp.z, wp.w)));
            const float2 c = cs2[p][i], s = sn2[p][i];
            const float2 ro = round16f2<BF16>(fma2(mul2(v, s), mone2, mul2(u, c)));  // u c - v s
            const float2 rv = round16f2<BF16>(fma2(mul2(u, s), one2, mul2(v, c)));   // u s + v c
            if constexpr (RM == kRotAll) {
                sink(p, i, ro, rv);
            } else if constexpr (RM == kRotFirst) {
                sink(p, i, make_float2(ro.x, rot1 ? ro.y : u.y), make_float2(rv.x, rot1 ? rv.y : v.y));
            } else {
                sink(p, i, make_float2(rot[2 * p][i] ? ro.x : u.x, rot[2 * p + 1][i] ? ro.y : u.y),
                     make_float2(rot[2 * p][i] ? rv.x : v.x, rot[2 * p + 1][i] ? rv.y : v.y));
            }
        }
}

// The cast of one Q/K head row on packed pairs: e4m3 codes of chunk q in
// code[q] (channels 0..7, lowest byte first), from the results of
// qk_row_pairs times the factor f2 (one rounded packed product).  With
// COUNT, the values of the chunks with act[q] set whose scaled magnitude
// exceeds 448 are added to sat.
template <bool BF16, int LPR, int CH, bool COUNT, int RM>
__device__ __forceinline__ void qk_row_pairs_e4m3(const uint4 (&raw)[CH], const float2* w2,
                                                  const float2 (&cs2)[CH / 2][4], const float2 (&sn2)[CH / 2][4],
                                                  const bool (&rot)[CH][4], bool rot1, float inv_d, float eps, int D,
                                                  float2 one2, float2 mone2, float2 f2, const bool (&act)[CH],
                                                  uint2 (&code)[CH], unsigned int& sat)
{
    uint32_t c16[CH][4];
    qk_row_pairs<BF16, LPR, CH, RM>(raw, w2, cs2, sn2, rot, rot1, inv_d, eps, D, one2, mone2,
                                [&](int p, int i, float2 yu, float2 yv) {
                                    const float2 zu = mul2(yu, f2), zv = mul2(yv, f2);
                                    c16[2 * p][i] = e4m3x2(zu.x, zv.x);
                                    c16[2 * p + 1][i] = e4m3x2(zu.y, zv.y);
                                    if constexpr (COUNT)
                                        sat += (act[2 * p] ? (fabsf(zu.x) > 448.0f) + (fabsf(zv.x) > 448.0f) : 0) +
                                               (act[2 * p + 1] ? (fabsf(zu.y) > 448.0f) + (fabsf(zv.y) > 448.0f)
                                                               : 0);
                                });
#pragma unroll
    for (int q = 0; q < CH; ++q) code[q] = make_uint2(c16[q][0] | (c16[q][1] << 16), c16[q][2] | (c16[q][3] << 16));
}

// The largest |y| over the chunks with act[q] set of one Q/K head row on
// packed pairs (NaN ignored), folded into m (a non-negative binary32).
template <bool BF16, int LPR, int CH, int RM>
__device__ __forceinline__ float qk_row_pairs_amax(const uint4 (&raw)[CH], const float2* w2,
                                                   const float2 (&cs2)[CH / 2][4], const float2 (&sn2)[CH / 2][4],
                                                   const bool (&rot)[CH][4], bool rot1, float inv_d, float eps, int D,
                                                   float2 one2, float2 mone2, const bool (&act)[CH], float m)
{
    qk_row_pairs<BF16, LPR, CH, RM>(raw, w2, cs2, sn2, rot, rot1, inv_d, eps, D, one2, mone2,
                                [&](int p, int i, float2 yu, float2 yv) {
                                    if (act[2 * p]) m = fmaxf(m, fmaxf(fabsf(yu.x), fabsf(yv.x)));
                                    if (act[2 * p + 1]) m = fmaxf(m, fmaxf(fabsf(yu.y), fabsf(yv.y)));
                                });
    return m;
}

// The same head row for the sage outputs: every step stays binary32 (the
// normalised value is not rounded to 16 bits before the rotation), and the
// lane's CH*8 results are returned unrounded, chunk by chunk.
template <bool BF16, int LPR, int CH>
__device__ __forceinline__ void qk_row_f32(const uint4 (&raw)[CH], const float4* w, const float (&cs)[CH][4],
                                           const float (&sn)[CH][4], const bool (&rot)[CH][4], float inv_d,
                                           float eps, int D, float (&y)[CH][8])
{
    float x[CH][8];
    const float inv = qk_inv<BF16, LPR, CH>(raw, inv_d, eps, D, x);
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int q = 0; q < CH; ++q) {
        const float4 wa = w[2 * q], wb = w[2 * q + 1];
        const float wq[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = mul2(mul2(make_float2(x[q][2 * i], x[q][2 * i + 1]), inv2),
                                  make_float2(wq[2 * i], wq[2 * i + 1]));
            const float ro = __fsub_rn(__fmul_rn(a.x, cs[q][i]), __fmul_rn(a.y, sn[q][i]));  // u c - v s
            const float rv = __fadd_rn(__fmul_rn(a.x, sn[q][i]), __fmul_rn(a.y, cs[q][i]));  // u s + v c
            y[q][2 * i] = rot[q][i] ? ro : a.x;
            y[q][2 * i + 1] = rot[q][i] ? rv : a.y;
        }
    }
}

// Eight binary32 values (optionally times k) -> two 16-byte stores at dst.
__device__ __forceinline__ void store_f32x8(const float (&y)[8], float k, bool scale, float* dst)
{
    float2 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = make_float2(y[2 * i], y[2 * i + 1]);
        if (scale) v[i] = mul2(v[i], make_float2(k, k));
    }
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
}

// Eight 16-bit values times k, each product rounded to binary32 and then to
// binary16 (nearest even, overflow to infinity): one 16-byte store at dst.
template <bool BF16>
__device__ __forceinline__ void store_v_f16(const uint4& raw, float k, uint16_t* dst)
{
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 z = mul2(widen2<BF16>(word(raw, i)), make_float2(k, k));
        __half2 h = __floats2half2_rn(z.x, z.y);
        o[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Upper bound on |y| over one Q/K head row slice (amax pass early-out).
// Every 16-bit output y of the row satisfies
//   |y| <= sqrt(2) (1 + 2^-8)^2 (1 + 2^-22) max|x| max|w| inv + 2^-24
//       <= 1.4253 max|x| max|w| inv + 2^-24:
// a rotated pair obeys |u c - v s| <= sqrt(u^2 + v^2) sqrt(c^2 + s^2) with
// c^2 + s^2 <= 1 + 7e-7 (the sine/cosine error bound), each of the two
// 16-bit roundings adds at most 2^-8 relative (plus half a subnormal step),
// the binary32 products and sums 2^-24 each.  The bound evaluates inv from an
// approximate sum of squares (fused multiply-adds, any order) and rsqrtf,
// within 2^-19 relative of the exact inv, and takes 1.45 and 2^-23, a margin
// of 1.7 % over the exact bound.  max|x| comes from the packed 16-bit inputs
// (exact), max|w| is the lane's largest weight.  A NaN or infinite input gives
// a NaN or infinite bound, which never allows a skip.  So does an approximate
// sum of squares at or above 2^126: near the binary32 overflow the two
// summation orders may round to different sides of FLT_MAX, and an infinite
// approximate sum would otherwise give inv = 0 and a bound of 2^-23 for a row
// whose exact values are not small.  Below 2^126 the exact sum cannot
// overflow, and the error analysis above holds.  At the other end, a sum
// under the root (ss/D + eps) below 2^-96 also gives an infinite bound: with
// eps = 0 and squares in the binary32 subnormal range, the two orders can
// differ by a subnormal quantum, a large relative error when the whole sum is
// a few quanta (and a rotated pair of such a row reaches ordinary sizes).
// Above 2^-96 those absolute differences are below 2^-40 relative.
// bfloat16 inputs accumulate their squares as packed bfloat16 fused
// multiply-adds on the input words (no widening): each of the 4*CH steps per
// half rounds up by at most 2^-8 relative, so the sum is at most
// (1 + 2^-8)^(4 CH) above the exact one (below it is the safe side), inv at
// most (1 + 2^-8)^(2 CH) below, and the constant grows to 1.47 for CH = 2
// (1.45 for CH = 1, 1.49 for CH = 4), again with about 1.5 % to spare.  An
// overflowing or vanishing packed sum meets the two guards above.
// The sum under the root that the bound used goes to `t` (left unset when
// the bound is infinite).
template <bool BF16, int LPR, int CH>
__device__ __forceinline__ float qk_bound(const uint4 (&raw)[CH], float wmax, float inv_d, float eps, int D,
                                          float& t_out)
{
    uint32_t m2 = 0u;
    float ss;
    if constexpr (BF16) {
        uint32_t acc = 0u;  // two bfloat16 partial sums
#pragma unroll
        for (int q = 0; q < CH; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w = word(raw[q], i);
                m2 = hmax2x<true>(m2, w);
                __nv_bfloat162 r = __hfma2(*reinterpret_cast<__nv_bfloat162*>(&w),
                                           *reinterpret_cast<__nv_bfloat162*>(&w),
                                           *reinterpret_cast<__nv_bfloat162*>(&acc));
                acc = *reinterpret_cast<uint32_t*>(&r);
            }
        const float2 a = widen2<true>(acc);
        ss = a.x + a.y;
    } else {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < CH; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = word(raw[q], i);
                m2 = hmax2x<false>(m2, w);
                const float2 x = widen2<false>(w);
                acc = __ffma2_rn(x, x, acc);
            }
        ss = acc.x + acc.y;
    }
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (!(ss < 0x1p126f)) return __int_as_float(0x7f800000);  // +inf: never skip
    const float t = ss * (inv_d != 0.0f ? inv_d : 1.0f / static_cast<float>(D)) + eps;
    if (!(t >= 0x1p-96f)) return __int_as_float(0x7f800000);  // +inf: never skip
    t_out = t;
    const float inv = rsqrtf(t);
    constexpr float kMargin = !BF16 ? 1.45f : (CH == 1 ? 1.45f : (CH == 2 ? 1.47f : 1.49f));
    return kMargin * inv * hmax2x_to_float<BF16>(m2) * wmax + 0x1p-23f;
}

// Second, tighter test of the early-out, for rows whose first bound did not
// allow a skip: true when some |y| of this lane's row slice may exceed
// `known` (an exact |y| already seen).  With z_j = x_j w_j, every output of
// a channel pair (j, j+1) obeys
//   |y| <= (1 + u)^2 (1 + 2^-24)^4 sqrt(1 + 7e-7) inv sqrt(z_j^2 + z_{j+1}^2) + 3 a
// (u = 2^-8 for bfloat16, 2^-11 for float16; a = half the 16-bit subnormal
// step): the same steps as above with the rotation bounded by the pair's own
// norm instead of sqrt(2) max|x| max|w| (a pair that is not rotated keeps one
// of its two values, below the norm as well).  Squared and compared with
// t = ss/D + eps from the first bound, no root or division is taken: skip
// when K2 max_j(z_j^2 + z_{j+1}^2) <= known^2 t.  K2 covers (1 + u)^4, the
// sine/cosine term, the binary32 steps on both sides (below 2^-16 together),
// the approximate sum in t (bfloat16: up to (1 + 2^-8)^(4 CH) above the
// exact one; float16: under 2^-19), and (1 + 2^-9)^2, which absorbs the
// absolute term once known >= 2^-13 (3a <= 2^-23 <= 2^-10 known).  That gives
// 1.0359, 1.0522 and 1.0856 for bfloat16 with CH = 1, 2, 4 and 1.0059 for
// float16, taken as 1.04, 1.06, 1.09 and 1.01.  known above 2^60 (its
// square could overflow) or below 2^-13 never allows a skip.  Nor does a
// NaN or infinite pair square (from a NaN or infinite weight; the inputs are
// finite once the first bound is): the maximum keeps a NaN, and the
// comparison is then false.  An overflowing right-hand side is safe: its
// exact value then exceeds every finite left-hand side.
__device__ __forceinline__ float fmax_keep_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

template <bool BF16, int CH>
__device__ __forceinline__ bool qk_pair_may_exceed(const uint4 (&raw)[CH], const float4* w, float t, float known)
{
    float m = 0.0f;
#pragma unroll
    for (int q = 0; q < CH; ++q) {
        const float4 wa = w[2 * q], wb = w[2 * q + 1];
        const float wq[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 z = mul2(widen2<BF16>(word(raw[q], i)), make_float2(wq[2 * i], wq[2 * i + 1]));
            m = fmax_keep_nan(m, __fmaf_rn(z.x, z.x, __fmul_rn(z.y, z.y)));
        }
    }
    if (!(known >= 0x1p-13f && known <= 0x1p60f)) return true;
    constexpr float kK2 = !BF16 ? 1.01f : (CH == 1 ? 1.04f : (CH == 2 ? 1.06f : 1.09f));
    const float lhs = kK2 * m;
    return !(lhs < 0x1p127f && lhs <= known * known * t);
}

// qk_pair_may_exceed for the weights in pair layout (float2 {w(chunk 2p, k),
// w(chunk 2p+1, k)} at [p*8 + k]): the same pair squares, two chunks per
// packed operation.
template <bool BF16, int CH>
__device__ __forceinline__ bool qk_pair_may_exceed2(const uint4 (&raw)[CH], const float2* w2, float t, float known)
{
    float m = 0.0f;
#pragma unroll
    for (int p = 0; p < CH / 2; ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 wp = reinterpret_cast<const float4*>(w2)[p * 4 + i];
            const float2 a = widen2<BF16>(word(raw[2 * p], i));
            const float2 b = widen2<BF16>(word(raw[2 * p + 1], i));
            const float2 zu = mul2(make_float2(a.x, b.x), make_float2(wp.x, wp.y));
            const float2 zv = mul2(make_float2(a.y, b.y), make_float2(wp.z, wp.w));
            const float2 sq = fma2(zu, zu, mul2(zv, zv));
            m = fmax_keep_nan(m, fmax_keep_nan(sq.x, sq.y));
        }
    if (!(known >= 0x1p-13f && known <= 0x1p60f)) return true;
    constexpr float kK2 = !BF16 ? 1.01f : (CH == 1 ? 1.04f : (CH == 2 ? 1.06f : 1.09f));
    const float lhs = kK2 * m;
    return !(lhs < 0x1p127f && lhs <= known * known * t);
}

// Eight 16-bit values -> eight e4m3 codes at dst (8 bytes); with COUNT, adds
// the number of values whose scaled magnitude exceeds 448 (clipped to the
// largest code) to sat.
template <bool BF16, bool COUNT>
__device__ __forceinline__ void emit_e4m3(const uint32_t (&y)[4], float f, uint8_t* dst, unsigned int& sat)
{
    const float2 fa = make_float2(f, f);
    uint32_t cw[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 z0 = mul2(widen2<BF16>(y[2 * i]), fa);
        const float2 z1 = mul2(widen2<BF16>(y[2 * i + 1]), fa);
        cw[i] = e4m3x2(z0.x, z0.y) | (e4m3x2(z1.x, z1.y) << 16);
        if constexpr (COUNT)
            sat += (fabsf(z0.x) > 448.0f) + (fabsf(z0.y) > 448.0f) + (fabsf(z1.x) > 448.0f) +
                   (fabsf(z1.y) > 448.0f);
    }
    *reinterpret_cast<uint2*>(dst) = make_uint2(cw[0], cw[1]);
}

// ---------------------------------------------------------------------------
// The kernel.  A head row's C = D/8 chunks (8 channels = 16 bytes each) sit on
// LPR lanes, CH chunks per lane: lane c owns chunks c, c + LPR, ..., with
// LPR * CH = P = next_pow2(C).  A warp covers TPW = 32/LPR token rows.  Each
// warp walks groups of TPW rows (grid-stride) and, for each, the H head rows
// of Q, then of K (norm + RoPE), then of V (copied), U head rows per batch of
// loads; a call on one tensor runs only its own part.  Outputs go to
// item * out_bstride + token * out_sstride + head * out_hstride (head-major
// [B, H, S, D] or token-major [B, S, H, D]).  The reduction tree is the same for every (LPR, CH): the first
// halving level (chunk c + chunk c+LPR) is in-lane, the rest are xor shuffles.
// MODE kOut16 writes 16-bit head-major outputs; kAmax reduces max |y| per
// tensor; kCast writes e4m3 codes under the dynamic or static factors, and
// kCastCount does the same and adds the clipped-value counts; kSage writes
// binary32 Q, binary32 K * kv_scale and binary16 V * kv_scale.
// ---------------------------------------------------------------------------
// Item (batch index) of token row r < p.rows: r / seq, without a division
// when the call has one item, and in 32 bits when the rows fit.
__device__ __forceinline__ int64_t item_of(const Params& p, int64_t r)
{
    if (p.rows == p.seq) return 0;
    if (p.rows <= 0x7fffffff) return static_cast<int64_t>(static_cast<uint32_t>(r) / static_cast<uint32_t>(p.seq));
    return r / p.seq;
}

// Lane groups of a warp that share a token row (the amax head split, see HS
// in the kernel), and the token rows of one work item.
template <int MODE, int LPR>
__host__ __device__ constexpr int head_split()
{
    return MODE == kAmax && (32 / LPR) % H3QK_AMAX_HEAD_SPLIT == 0 ? H3QK_AMAX_HEAD_SPLIT : 1;
}
template <int MODE, int LPR>
__host__ __device__ constexpr int rows_per_item()
{
    return 32 / LPR / head_split<MODE, LPR>();
}

template <bool BF16, int LPR, int CH, int MODE, bool SLICED, int RM>
__global__ void __launch_bounds__(Shape<MODE, LPR>::NT, Shape<MODE, LPR>::MB)
    qkprep_kernel(const __grid_constant__ Params p)
{
    static_assert(CH == 1 || CH == 2 || CH == 4, "1, 2 or 4 chunks per lane");
    constexpr int TPW = 32 / LPR;
    constexpr int U = TuneL<MODE, LPR>::U;    // Q/K head rows per batch of loads
    constexpr int S = TuneL<MODE, LPR>::S;    // shared-memory pipeline stages (0 = none)
    constexpr int UV = S > 0 ? U : TuneL<MODE, LPR>::UV;  // V head rows per batch (copy only)
    constexpr int PF = TuneL<MODE, LPR>::PF;  // L2 prefetch distance in batches
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    // Head split (amax): the warp's TPW lane groups take RPG token rows, HS
    // groups per row; group sub takes row sub / HS and, in each batch of HS*U
    // head rows, the U heads from (sub % HS)*U.  A batch then reads HS*U
    // consecutive head rows of each of its token rows (longer pieces of DRAM
    // at a time) with the same copies per lane.
    constexpr int HS = head_split<MODE, LPR>();
    constexpr int RPG = rows_per_item<MODE, LPR>();
    constexpr int HU = HS * U;   // head rows per batch and token row
    const int srow = sub / HS;
    const int hph = (sub % HS) * U;
    const int c = lane % LPR;
    bool on[CH];
#pragma unroll
    for (int q = 0; q < CH; ++q) on[q] = c + q * LPR < p.chunks;
    const int H = p.heads;
    const int D = p.head_dim;
    constexpr bool kCastMode = MODE == kCast || MODE == kCastCount;
    constexpr bool count_sat = MODE == kCastCount;
    // The e4m3 modes compute their Q/K rows on packed pairs of chunks (qk_row_pairs).
    constexpr bool kPairs = (kCastMode || MODE == kAmax) && CH >= 2;
    // Which channels rotate is a property of the call (RM, a RotMode chosen
    // at launch by rot_mode_of): all of them; the first chunk of every lane
    // and the second chunk of the lanes where rot1 is set; or any pattern.
    static_assert(RM == kRotAny || kPairs, "rotation modes other than kRotAny: e4m3 pair instances only");
    const bool rot1 = CH == 2 && 8 * (c + LPR) + 8 <= p.rotary_dim;
    const int64_t n_groups = (p.rows + RPG - 1) / RPG;
    // Work items: a row group, or (SLICED, for calls too small to fill the
    // GPU) one of 2^hs_shift slices of hs_heads heads of a row group.
    const int hs_shift = SLICED ? p.hs_shift : 0;
    const int64_t n_items = n_groups << hs_shift;
    const int hs_mask = (1 << hs_shift) - 1;
    // Row group of work item it.  The cast of a dynamic call walks the groups
    // from the last one down: its amax pass (the kernel just before it, which
    // only reads) walked them upwards, so the input rows it read last are
    // still in L2 and the cast reads those first.
    const bool rev = kCastMode && p.reverse != 0;
    auto group_of = [&](int64_t item) {
        const int64_t g0 = item >> hs_shift;
        return rev ? n_groups - 1 - g0 : g0;
    };
    // The amax pass walks each work item backwards: V, then K, then Q, each
    // from its last batch of heads down.  What it reads last in an item is
    // then what the cast (reversed groups, forward within an item) reads
    // first, so the cast's first reads hit the lines the amax pass left in
    // L2.  The maximum does not depend on the order.
    constexpr bool kBack = MODE == kAmax && H3QK_AMAX_BACK;
    // The kRotFirst cast instances (the ones closest to their register cap:
    // each value of a second chunk keeps its unrotated form until the choice)
    // keep a row group's rotary cos/sin in shared memory, per warp
    // [pair slot i][lane] as {cos chunk 0, cos chunk 1, sin chunk 0, sin
    // chunk 1}: four 16-byte loads per head row instead of 16 registers held
    // across the group, which halves their spills.
    constexpr bool kAngSmem = kCastMode && kPairs && CH == 2 && RM == kRotFirst && H3QK_SMEM_ANGLES;
    __shared__ __align__(16) float4 ang_store[kAngSmem ? Shape<MODE, LPR>::W * 4 * 32 : 1];
    float4* const angs = ang_store + (kAngSmem ? (threadIdx.x >> 5) * 4 * 32 : 0);
    constexpr int NT = Shape<MODE, LPR>::NT;  // threads per block
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * NT + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * NT) >> 5;

    // Chained launches.  A dynamic call runs three kernels: zero the amax
    // words, the amax pass, the cast.  The second and third are launched as
    // programmatic dependents of the one before (griddepcontrol), so each
    // is scheduled while its predecessor drains and stages its weights and
    // its first input copies meanwhile; it waits for the predecessor to
    // complete, with its writes visible, before it touches the amax words
    // (the amax pass before its first read of them, the cast before it
    // derives its factors).  Nothing before the wait reads or writes memory
    // that the predecessor writes, and the first kernel of a call is never
    // chained, so the inputs are complete when any kernel of the call
    // starts.  Outside a chained launch the wait returns at once.  The amax
    // pass lets its dependent (the cast) be scheduled from its start: the
    // cast's blocks only take SM room that finished amax blocks leave.
    if constexpr (MODE == kAmax) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Norm weights of Q and K in shared memory, laid out per lane:
    // ws[part][c][q*8 + k] = weight of channel 8*(c + q*LPR) + k (zero past
    // the head), so a lane reads its CH*8 weights as 2*CH float4.  The pair
    // layout of the casts interleaves chunks 2p and 2p+1 instead:
    // ws[part][c][p*16 + 2*k + j] = weight of channel k of chunk 2p+j.
    __shared__ __align__(16) float ws[2][LPR][CH * 8];
    for (int t = threadIdx.x; t < 2 * LPR * CH * 8; t += NT) {
        const int part = t / (LPR * CH * 8), cc = (t / (CH * 8)) % LPR, q = (t / 8) % CH, k = t % 8;
        const float* w = part == 0 ? p.wq : p.wk;
        const int chunk = cc + q * LPR;
        const bool used = part >= p.qk_first && part < p.qk_end;  // a V-only call has no weights
        const int at = kPairs ? (q / 2) * 16 + 2 * k + (q % 2) : q * 8 + k;
        ws[part][cc][at] = used && chunk < p.chunks ? __ldg(w + 8 * chunk + k) : 0.0f;
    }
    __syncthreads();
    // Largest |weight| of this lane per part (the amax pass's row bound).
    float wmax[2] = {0.0f, 0.0f};
    if constexpr (MODE == kAmax) {
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int k = 0; k < CH * 8; ++k) wmax[part] = fmaxf(wmax[part], fabsf(ws[part][c][k]));
    }
    // Warp-uniform running max of the exact |y| seen per part (binary32 bits),
    // the part of it already published to the amax words, and the published
    // grid-wide value read at the start of each part.  Every published value
    // is an exact |y| of some element, so it never exceeds the final amax and
    // rows bounded below it cannot change the result.
    uint32_t run[3] = {0u, 0u, 0u};
    uint32_t pub[2] = {0u, 0u};
    uint32_t thr[2] = {0u, 0u};

    uint32_t am[3] = {0u, 0u, 0u};  // packed 16-bit running max of |y| per tensor (hmax2x)
    float amf[2] = {0.0f, 0.0f};    // pair path: running max of |y| of Q and K
    unsigned int sat[3] = {0u, 0u, 0u};

    // ---- shared-memory pipeline (S > 0) -------------------------------------
    // Each lane copies its own 16-byte chunks of the batch S-1 steps ahead
    // into its warp's ring of S stages, walking the same sequence of batches
    // the loop below consumes (groups, then parts Q, K, V, then head
    // batches; kBack: parts V, K, Q and head batches from the last one
    // down); stage layout [S][U][CH][32 lanes] of uint4.
    extern __shared__ __align__(16) uint4 h3qk_stage[];
    uint4* const ring = h3qk_stage + static_cast<size_t>(threadIdx.x >> 5) * (S > 0 ? S * U * CH * 32 : 0);
    const bool has_qk = p.qk_first < p.qk_end;
    const int first_part = kBack ? (p.has_v || !has_qk ? 2 : p.qk_end - 1) : (has_qk ? p.qk_first : 2);
    int64_t fit = warp0;         // issue cursor: work item, part, head, stage
    int fpart = first_part, fh0 = 0, fh_lo = 0, fh_hi = H, fstage = 0;
    const uint16_t* frow = p.qkv;
    bool fact[CH];
    auto feed_group = [&]() {    // head slice, row pointer and active chunks of item fit
        if constexpr (SLICED) {
            fh_lo = static_cast<int>(fit & hs_mask) * p.hs_heads;
            fh_hi = min(H, fh_lo + p.hs_heads);
        }
        fh0 = kBack ? fh_lo + (fh_hi - fh_lo - 1) / HU * HU : fh_lo;
        const int64_t rr = group_of(fit) * RPG + srow;
        bool ok = false;
        if (rr < p.rows) {
            const int64_t bb = item_of(p, rr);
            int64_t vl = p.valid_len;
            if (p.valid_lens && dbg_ok(p, bb < p.rows / p.seq, kDbgLengths, bb)) {
                vl = __ldg(p.valid_lens + bb);
                vl = vl < 0 ? 0 : (vl > p.seq ? p.seq : vl);
            }
            ok = rr - bb * p.seq < vl;
        }
        frow = ok ? p.qkv + rr * p.row_stride + 8 * c : p.qkv;
#pragma unroll
        for (int q = 0; q < CH; ++q) fact[q] = ok && on[q];
    };
    auto issue = [&]() {         // copies of the next batch, one commit group
        if constexpr (S > 0) {
            if (fit < n_items) {
                uint4* st = ring + fstage * (U * CH * 32);
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int q = 0; q < CH; ++q)
                        if (fh0 + hph + u < fh_hi && fact[q]) {
                            const uint16_t* src_u =
                                frow + p.in_part_off[fpart] + static_cast<int64_t>(fh0 + hph + u) * D + 8 * q * LPR;
                            if (dbg_in(p, src_u - p.qkv)) cp_async16(st + (u * CH + q) * 32 + lane, src_u);
                        }
                if constexpr (kBack) {
                    fh0 -= HU;
                    if (fh0 < fh_lo) {
                        fh0 = fh_lo + (fh_hi - fh_lo - 1) / HU * HU;
                        if (fpart == 2 && has_qk) {
                            fpart = p.qk_end - 1;
                        } else if (fpart < 2 && fpart > p.qk_first) {
                            --fpart;
                        } else {
                            fpart = first_part;
                            fit += n_warps;
                            if (fit < n_items) feed_group();
                        }
                    }
                } else {
                    fh0 += HU;
                    if (fh0 >= fh_hi) {
                        fh0 = fh_lo;
                        if (fpart < 2 && fpart + 1 < p.qk_end) {
                            ++fpart;
                        } else if (fpart < 2 && p.has_v) {
                            fpart = 2;
                        } else {
                            fpart = first_part;
                            fit += n_warps;
                            if (fit < n_items) feed_group();
                        }
                    }
                }
            }
            cp_async_commit();
            fstage = fstage + 1 == S ? 0 : fstage + 1;
        }
    };
    int pstage = 0;              // stage of the batch the loop consumes next
    if constexpr (S > 0) {
        // Chunks past the head are never copied: their slots are zeroed once
        // here and stay zero, which pads the reduction (each lane owns its
        // slots, so no other lane writes them).
#pragma unroll
        for (int q = 0; q < CH; ++q)
            if (!on[q])
                for (int k = 0; k < S * U; ++k) ring[(k * CH + q) * 32 + lane] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < CH; ++q) fact[q] = false;
        if (fit < n_items) feed_group();
#pragma unroll 1
        for (int k = 0; k < S - 1; ++k) issue();
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Cast factors (each thread derives them; block 0 publishes the descales),
    // read after the wait above.
    float fac[3] = {1.0f, 1.0f, 1.0f};
    if constexpr (kCastMode) {
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            if (p.slot[t] < 0) continue;
            // One load from whichever table this mode uses (never a NULL pointer).
            const float a = dbg_slot(p, p.slot[t]) ? __uint_as_float(__ldcg(p.scale_words + p.slot[t])) : 0.0f;
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
            if (blockIdx.x == 0 && threadIdx.x == 0 && dbg_slot(p, p.slot[t])) p.out_scales[p.slot[t]] = s;
        }
    }

    for (int64_t it = warp0; it < n_items; it += n_warps) {
        const int64_t g = group_of(it);
        const int h_lo = SLICED ? static_cast<int>(it & hs_mask) * p.hs_heads : 0;
        const int h_hi = SLICED ? min(H, h_lo + p.hs_heads) : H;
        const int64_t r = g * RPG + srow;
        int64_t b = 0, s = 0;
        bool act_row = false;
        if (r < p.rows) {
            b = item_of(p, r);
            s = r - b * p.seq;
            int64_t vl = p.valid_len;
            if (p.valid_lens && dbg_ok(p, b < p.rows / p.seq, kDbgLengths, b)) {
                vl = __ldg(p.valid_lens + b);
                vl = vl < 0 ? 0 : (vl > p.seq ? p.seq : vl);
            }
            act_row = s < vl;
        }
        bool act[CH];
#pragma unroll
        for (int q = 0; q < CH; ++q) act[q] = act_row && on[q];

        // Rotary cos / sin of this lane's pairs: pair i of chunk q is global
        // pair 4*(c + q*LPR) + i.  The amax pass evaluates them only when a
        // row of the group escapes the early-out (a warp-uniform decision).
        float cs[CH][4], sn[CH][4];
        bool rot[CH][4];
#pragma unroll
        for (int q = 0; q < CH; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                rot[q][i] = 2 * (4 * (c + q * LPR) + i) < p.rotary_dim;
                cs[q][i] = 1.0f;
                sn[q][i] = 0.0f;
            }
        auto angles = [&]() {
#pragma unroll
            for (int q = 0; q < CH; ++q)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int pair = 4 * (c + q * LPR) + i;
                    if (rot[q][i] && act[q]) {
                        const int64_t pi = r * p.n_axes + p.axis[pair];
                        const float pv = dbg_ok(p, pi >= 0 && pi < p.rows * p.n_axes, kDbgPositions, pi)
                                             ? static_cast<float>(__ldg(p.pos + pi))
                                             : 0.0f;
                        sincos_h3(__fmul_rn(pv, p.inv_freq[pair]), sn[q][i], cs[q][i]);
                    }
                }
            if constexpr (kAngSmem) {
#pragma unroll
                for (int i = 0; i < 4; ++i) angs[i * 32 + lane] = make_float4(cs[0][i], cs[1][i], sn[0][i], sn[1][i]);
            }
        };
        // The packed cos / sin of pair slot i for the pair code: from shared
        // memory (kAngSmem) or from the registers above.
        auto pair_angles = [&](float2 (&cs2)[CH / 2][4], float2 (&sn2)[CH / 2][4]) {
            if constexpr (kAngSmem) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 a = angs[i * 32 + lane];
                    cs2[0][i] = make_float2(a.x, a.y);
                    sn2[0][i] = make_float2(a.z, a.w);
                }
            } else {
#pragma unroll
                for (int pp = 0; pp < CH / 2; ++pp)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        cs2[pp][i] = make_float2(cs[2 * pp][i], cs[2 * pp + 1][i]);
                        sn2[pp][i] = make_float2(sn[2 * pp][i], sn[2 * pp + 1][i]);
                    }
            }
        };
        bool have_angles = MODE != kAmax;
        if constexpr (MODE != kAmax) angles();

        const uint16_t* rowp = p.qkv + r * p.row_stride + 8 * c;
        const int64_t obase = b * p.out_bstride + s * p.out_sstride + 8 * c;

        // L2 prefetch of this row's input PF batches ahead of the
        // batch starting at element `cur`; past the row's end it continues in
        // the row this lane handles next (grid stride).  One lane per row.
        auto prefetch = [&](int64_t cur, int64_t n) {
            if constexpr (PF > 0) {
                if (c != 0) return;
                int64_t off = cur + static_cast<int64_t>(PF) * n;
                int64_t rr = r;
                if (off >= p.pf_span) {
                    off -= p.pf_span;
                    rr = group_of(it + n_warps) * TPW + sub;
                }
                if (rr < 0 || rr >= p.rows || off >= p.pf_span) return;  // past the last item either way
                if (off + n > p.pf_span) n = p.pf_span - off;
                prefetch_l2(p.qkv + rr * p.row_stride + off, static_cast<uint32_t>(2 * n));
            }
        };

        // ---- V: passed through ----------------------------------------------
        auto v_part = [&]() {
            const uint16_t* src = rowp + p.in_part_off[2];
            constexpr int HUV = HS * UV;
            const int hv_first = kBack ? h_lo + (h_hi - h_lo - 1) / HUV * HUV : h_lo;  // first batch of heads
            for (int h0 = hv_first; kBack ? h0 >= h_lo : h0 < h_hi; h0 += kBack ? -HUV : HUV) {
                prefetch(p.in_part_off[2] + static_cast<int64_t>(h0) * D, static_cast<int64_t>(UV) * D);
                uint4 raw[UV][CH];
                if constexpr (S > 0) {
                    issue();
                    cp_async_wait<(S > 0 ? S - 1 : 0)>();
                    const uint4* st = ring + pstage * (U * CH * 32);
#pragma unroll
                    for (int u = 0; u < UV; ++u)
#pragma unroll
                        for (int q = 0; q < CH; ++q)
                            raw[u][q] = st[(u * CH + q) * 32 + lane];
                    pstage = pstage + 1 == S ? 0 : pstage + 1;
                } else {
#pragma unroll
                    for (int u = 0; u < UV; ++u)
#pragma unroll
                        for (int q = 0; q < CH; ++q) {
                            raw[u][q] = make_uint4(0u, 0u, 0u, 0u);
                            if (h0 + hph + u < h_hi && act[q]) {
                                const uint16_t* a = src + static_cast<int64_t>(h0 + hph + u) * D + 8 * q * LPR;
                                if (dbg_in(p, a - p.qkv)) raw[u][q] = load16(a);
                            }
                        }
                }
#pragma unroll
                for (int u = 0; u < UV; ++u) {
                    const int h = h0 + hph + u;
                    if (h >= h_hi) {
                        if constexpr (HS == 1) break;  // warp-uniform
                        else continue;  // head split (amax): no warp-wide step follows for V
                    }
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        if (!act[q]) continue;
                        const int64_t off = obase + h * p.out_hstride + 8 * q * LPR;
                        if constexpr (MODE == kOut16) {
                            uint16_t* dst = static_cast<uint16_t*>(p.out[2]) + off;
                            if (dbg_out(p, off)) *reinterpret_cast<uint4*>(dst) = raw[u][q];
                        } else if constexpr (MODE == kSage) {
                            if (dbg_out(p, off))
                                store_v_f16<BF16>(raw[u][q], p.kv_scale, static_cast<uint16_t*>(p.out[2]) + off);
                        } else if constexpr (MODE == kAmax) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) am[2] = hmax2x<BF16>(am[2], word(raw[u][q], i));
                        } else {
                            const uint32_t yv[4] = {raw[u][q].x, raw[u][q].y, raw[u][q].z, raw[u][q].w};
                            uint8_t* dst = static_cast<uint8_t*>(p.out[2]) + off;
                            if (dbg_out(p, off)) emit_e4m3<BF16, count_sat>(yv, fac[2], dst, sat[2]);
                        }
                    }
                }
            }
        };

        // ---- Q and K: norm + RoPE ------------------------------------------
        if constexpr (kBack) {
            if (p.has_v) v_part();
        }
#pragma unroll
        for (int pi = 0; pi < 2; ++pi) {
            const int part = kBack ? 1 - pi : pi;
            if (part < p.qk_first || part >= p.qk_end) continue;  // warp-uniform
            const uint16_t* src = rowp + p.in_part_off[part];
            const int h_first = kBack ? h_lo + (h_hi - h_lo - 1) / HU * HU : h_lo;  // first batch of heads
            for (int h0 = h_first; kBack ? h0 >= h_lo : h0 < h_hi; h0 += kBack ? -HU : HU) {
                prefetch(p.in_part_off[part] + static_cast<int64_t>(h0) * D, static_cast<int64_t>(U) * D);
                if constexpr (MODE == kAmax) {
                    // Once per part: re-reading every batch made the three amax
                    // words a hot spot for every warp of the grid.
                    if (h0 == h_first) {
                        const uint32_t gw =
                            lane == 0 && dbg_slot(p, p.slot[part]) ? __ldcg(p.amax_words + p.slot[part]) : 0u;
                        thr[part] = __shfl_sync(0xffffffffu, gw, 0);
                    }
                }
                uint4 raw[U][CH];
                if constexpr (S > 0) {
                    // Keep the ring S-1 batches ahead, then take this batch.  Only
                    // chunks past the head read as zero (their slots, zeroed at the
                    // start, pad the reduction); a
                    // padded row's or a missing head's slot holds stale bytes, which
                    // never reach a store, the amax or a count (every use is masked
                    // by act / the head loop, and the amax bound of such a row is 0).
                    issue();
                    cp_async_wait<(S > 0 ? S - 1 : 0)>();
                    const uint4* st = ring + pstage * (U * CH * 32);
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int q = 0; q < CH; ++q)
                            raw[u][q] = st[(u * CH + q) * 32 + lane];
                    pstage = pstage + 1 == S ? 0 : pstage + 1;
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int q = 0; q < CH; ++q) {
                            raw[u][q] = make_uint4(0u, 0u, 0u, 0u);
                            if (h0 + hph + u < h_hi && act[q]) {
                                const uint16_t* a = src + static_cast<int64_t>(h0 + hph + u) * D + 8 * q * LPR;
                                if (dbg_in(p, a - p.qkv)) raw[u][q] = load16(a);
                            }
                        }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int h = h0 + hph + u;
                    if constexpr (HS == 1) {
                        if (h >= h_hi) break;  // warp-uniform
                    }
                    // With a head split the lane groups of a warp take different
                    // heads, so a head past the slice is masked instead (the
                    // steps below are warp-wide).
                    const bool hrow = act_row && h < h_hi;
                    bool acth[CH];
#pragma unroll
                    for (int q = 0; q < CH; ++q) acth[q] = act[q] && h < h_hi;
                    uint4 rw[CH];
#pragma unroll
                    for (int q = 0; q < CH; ++q) rw[q] = raw[u][q];
                    if constexpr (MODE == kAmax) {
                        // Exact early-out: when no lane's bound exceeds the largest
                        // exact |y| known (this warp's, or the grid's published
                        // one), the row cannot raise the amax.
                        float t = 0.0f;
                        const float bnd = qk_bound<BF16, LPR, CH>(rw, wmax[part], p.inv_d, p.eps, D, t);
                        const uint32_t bb = hrow ? __float_as_uint(bnd) : 0u;
                        const uint32_t known = run[part] > thr[part] ? run[part] : thr[part];
                        if (__reduce_max_sync(0xffffffffu, bb) <= known) continue;  // warp-uniform
                        if constexpr (TPW >= H3QK_AMAX_PAIR_MIN_TPW) {
                            // Where the first vote fails (a head with an outlier
                            // channel fails it in every row), the pairwise test
                            // lets most rows skip the exact path.
                            bool may = hrow && !(bnd < 0x1p127f);
                            if constexpr (kPairs) {
                                may = may || (hrow && qk_pair_may_exceed2<BF16, CH>(
                                                             rw, reinterpret_cast<const float2*>(&ws[part][c][0]),
                                                             t, __uint_as_float(known)));
                            } else {
                                may = may || (hrow && qk_pair_may_exceed<BF16, CH>(
                                                             rw, reinterpret_cast<const float4*>(&ws[part][c][0]),
                                                             t, __uint_as_float(known)));
                            }
                            if (!__any_sync(0xffffffffu, may)) continue;  // warp-uniform
                        }
                        if (!have_angles) {
                            angles();
                            have_angles = true;
                        }
                    }
                    if constexpr (MODE == kSage) {
                        float yf[CH][8];
                        qk_row_f32<BF16, LPR, CH>(rw, reinterpret_cast<const float4*>(&ws[part][c][0]), cs, sn,
                                                  rot, p.inv_d, p.eps, D, yf);
#pragma unroll
                        for (int q = 0; q < CH; ++q) {
                            if (!act[q]) continue;
                            const int64_t off = obase + h * p.out_hstride + 8 * q * LPR;
                            if (dbg_out(p, off))
                                store_f32x8(yf[q], p.kv_scale, part == 1, static_cast<float*>(p.out[part]) + off);
                        }
                        continue;
                    }
                    if constexpr (kPairs && MODE == kAmax) {
                        float2 cs2[CH / 2][4], sn2[CH / 2][4];
                        pair_angles(cs2, sn2);
                        amf[part] = qk_row_pairs_amax<BF16, LPR, CH, RM>(
                            rw, reinterpret_cast<const float2*>(&ws[part][c][0]), cs2, sn2, rot, rot1, p.inv_d,
                            p.eps, D, p.one2, p.mone2, acth, amf[part]);
                        run[part] = __reduce_max_sync(0xffffffffu, __float_as_uint(amf[part]));
                        if (run[part] > pub[part]) {  // warp-uniform
                            if (lane == 0 && dbg_slot(p, p.slot[part])) atomicMax(p.amax_words + p.slot[part], run[part]);
                            pub[part] = run[part];
                        }
                        continue;
                    } else if constexpr (kPairs) {
                        float2 cs2[CH / 2][4], sn2[CH / 2][4];
                        pair_angles(cs2, sn2);
                        uint2 code[CH];
                        qk_row_pairs_e4m3<BF16, LPR, CH, count_sat, RM>(
                            rw, reinterpret_cast<const float2*>(&ws[part][c][0]), cs2, sn2, rot, rot1, p.inv_d,
                            p.eps, D, p.one2, p.mone2, make_float2(fac[part], fac[part]), act, code, sat[part]);
#pragma unroll
                        for (int q = 0; q < CH; ++q) {
                            if (!act[q]) continue;
                            const int64_t off = obase + h * p.out_hstride + 8 * q * LPR;
                            if (dbg_out(p, off))
                                *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out[part]) + off) = code[q];
                        }
                        continue;
                    }
                    uint32_t y[CH][4];
                    qk_row<BF16, LPR, CH>(rw, reinterpret_cast<const float4*>(&ws[part][c][0]), cs, sn, rot,
                                          p.inv_d, p.eps, D, y);
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        if (!acth[q]) continue;
                        const int64_t off = obase + h * p.out_hstride + 8 * q * LPR;
                        if constexpr (MODE == kOut16) {
                            uint16_t* dst = static_cast<uint16_t*>(p.out[part]) + off;
                            if (dbg_out(p, off))
                                *reinterpret_cast<uint4*>(dst) = make_uint4(y[q][0], y[q][1], y[q][2], y[q][3]);
                        } else if constexpr (MODE == kAmax) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) am[part] = hmax2x<BF16>(am[part], y[q][i]);
                        } else {
                            uint8_t* dst = static_cast<uint8_t*>(p.out[part]) + off;
                            if (dbg_out(p, off)) emit_e4m3<BF16, count_sat>(y[q], fac[part], dst, sat[part]);
                        }
                    }
                    if constexpr (MODE == kAmax) {
                        run[part] = __reduce_max_sync(0xffffffffu, __float_as_uint(hmax2x_to_float<BF16>(am[part])));
                        if (run[part] > pub[part]) {  // warp-uniform
                            if (lane == 0 && dbg_slot(p, p.slot[part])) atomicMax(p.amax_words + p.slot[part], run[part]);
                            pub[part] = run[part];
                        }
                    }
                }
            }
        }
        if constexpr (!kBack) {
            if (p.has_v) v_part();
        }
    }

    if constexpr (S > 0) cp_async_wait<0>();  // only empty groups remain; keep the exit clean

    if constexpr (MODE == kAmax) {
        __shared__ float red[3][Shape<MODE, LPR>::W];
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            float m = hmax2x_to_float<BF16>(am[t]);
            if (kPairs && t < 2) m = amf[t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) red[t][threadIdx.x >> 5] = m;
        }
        __syncthreads();
        if (threadIdx.x < 3 && p.slot[threadIdx.x] >= 0) {
            float m = 0.0f;
#pragma unroll
            for (int w = 0; w < Shape<MODE, LPR>::W; ++w) m = fmaxf(m, red[threadIdx.x][w]);
            // Non-negative binary32 values order like their bit patterns.
            if (m > 0.0f && dbg_slot(p, p.slot[threadIdx.x]))
                atomicMax(p.amax_words + p.slot[threadIdx.x], __float_as_uint(m));
        }
    }
    if constexpr (count_sat) {
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            unsigned int n = sat[t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
            if (lane == 0 && n > 0 && p.slot[t] >= 0 && dbg_slot(p, p.slot[t])) atomicAdd(p.sat_counts + p.slot[t], n);
        }
    }
}


// The rotation mode (RotMode) of a call with rotary width R and head_dim D
// on an instance with LPR lanes and CH chunks per lane: every channel
// rotates (R == D); every lane's first chunk rotates and second chunks rotate
// whole or not at all (two chunks per lane, R a multiple of 8 covering the
// first LPR chunks); else any pattern.
__host__ __device__ constexpr int rot_mode_of(int R, int D, int LPR, int CH)
{
    return R == D ? kRotAll
                  : ((CH == 2 && LPR >= H3QK_ROT_FIRST_MIN_LPR && R % 8 == 0 && R >= 8 * LPR) ? kRotFirst : kRotAny);
}

}  // namespace h3qk
