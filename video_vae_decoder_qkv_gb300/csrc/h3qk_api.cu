// Host side of libh3qk: argument checks, rotary tables and the device entry
// points of the C-ABI declared in include/h3qk.h.  The kernel instances live
// in h3qk_launch_bf16.cu / h3qk_launch_fp16.cu, the host-buffer entry point
// in h3qk_host.cu.
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "h3qk.h"
#include "h3qk_internal.h"
#include "h3qk_kernels.cuh"

namespace h3qk {

// Zero the three amax words of a dynamic call (defined here only: this is
// the one translation unit that launches it).
__global__ void amax_init_kernel(unsigned int* words)
{
    // The amax pass that follows is a chained launch (it waits for this
    // kernel to complete before it reads the words).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x < 3) words[threadIdx.x] = 0u;
}

}  // namespace h3qk

namespace {

thread_local int g_last_cuda_error = 0;
thread_local uint64_t g_launches = 0;

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};

// Streaming multiprocessors of the current device (cached per device).
int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
    if (dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    if (dev < kMaxDevices) g_sm_count[dev] = n;
    return n;
}

int next_pow2(int v)
{
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

h3qk_status fail_cuda(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    return H3QK_ERR_CUDA;
}

}  // namespace

// ---------------------------------------------------------------------------
// Debug builds: the status words of the kernels' bounds checks (dbg_ok in
// h3qk_kernels.cuh), one set per device, and a test hook that narrows the
// output extent the checks allow.
// ---------------------------------------------------------------------------
#if H3QK_DEBUG_CHECKS
static __device__ __align__(16) unsigned int g_dbg_status[4];
#endif
namespace {
std::mutex g_dbg_mu;
#if H3QK_DEBUG_CHECKS
unsigned int* g_dbg_addr[kMaxDevices] = {nullptr};
#endif
int64_t g_dbg_out_limit = -1;  // < 0: the call's own output extent
}  // namespace

// Device address of the status words on the current device (null in release
// builds or when it cannot be looked up; the checks then only skip).
static unsigned int* dbg_status_addr()
{
#if H3QK_DEBUG_CHECKS
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_dbg_mu);
    if (!g_dbg_addr[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_dbg_status) != cudaSuccess) return nullptr;
        g_dbg_addr[dev] = static_cast<unsigned int*>(a);
    }
    return g_dbg_addr[dev];
#else
    return nullptr;
#endif
}

int h3qk_internal_sm_count() { return sm_count(); }
void h3qk_internal_count_launch() { ++g_launches; }
h3qk_status h3qk_internal_fail_cuda(cudaError_t e) { return fail_cuda(e); }

extern "C" {

void h3qk_opts_init(h3qk_opts* o)
{
    if (!o) return;
    std::memset(o, 0, sizeof(*o));
    o->in_dtype = H3QK_DTYPE_DEFAULT;
    o->n_axes = 3;
    o->eps = 1e-6f;
    o->batch = 1;
    o->qkv_row_stride = 0;
    o->theta = 10000.0;
    o->out_layout = H3QK_LAYOUT_HEAD_MAJOR;
    o->valid_lens = nullptr;
    o->sat_counts = nullptr;
}

size_t h3qk_workspace_bytes(void) { return 16; }

const char* h3qk_status_string(h3qk_status s)
{
    switch (s) {
    case H3QK_OK: return "ok";
    case H3QK_ERR_INVALID_ARG: return "invalid argument";
    case H3QK_ERR_MISALIGNED: return "misaligned pointer or row stride";
    case H3QK_ERR_ALIAS: return "an output overlaps an input or another output";
    case H3QK_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

int h3qk_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t h3qk_launch_count(void) { return g_launches; }

void h3qk_launch_count_reset(void) { g_launches = 0; }

int h3qk_version(void) { return 101; }

int h3qk_debug_checks(void) { return H3QK_DEBUG_CHECKS ? 1 : 0; }

h3qk_status h3qk_debug_status(uint32_t* out, int reset)
{
    if (!out || !H3QK_DEBUG_CHECKS) return H3QK_ERR_INVALID_ARG;
    unsigned int* a = dbg_status_addr();
    if (!a) return h3qk_internal_fail_cuda(cudaErrorInvalidSymbol);
    cudaError_t e = cudaMemcpy(out, a, 16, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && reset) e = cudaMemset(a, 0, 16);
    return e == cudaSuccess ? H3QK_OK : h3qk_internal_fail_cuda(e);
}

void h3qk_debug_limit_outputs(int64_t elements)
{
    std::lock_guard<std::mutex> lock(g_dbg_mu);
    g_dbg_out_limit = elements;
}

}  // extern "C"

namespace h3qk_detail {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

Range range_of(const void* p, int64_t bytes)
{
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes > 0 ? bytes : 0)};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

cudaError_t launch(bool bf16, int P, int mode, const h3qk::Params& p, cudaStream_t st)
{
    // A cast that counts clipped values runs its own instance.
    if (mode == h3qk::kCast && p.sat_counts) mode = h3qk::kCastCount;
    return bf16 ? h3qk_internal_launch_bf16(P, mode, p, st) : h3qk_internal_launch_fp16(P, mode, p, st);
}


// Checks of everything that describes the input rows (sizes, options, input
// pointers and their alignment) and the launch plan.  `default_in` is the
// input type assumed when opts->in_dtype is DEFAULT.
h3qk_status plan_inputs(const void* qkv, const float* norm_wq, const float* norm_wk,
                        const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                        int32_t rotary_dim, int64_t valid_len, int default_in, const h3qk_opts& o,
                        h3qk_stream_t stream, Plan* plan, int parts)
{
    if (tokens < 0 || heads < 1 || heads > 65536) return H3QK_ERR_INVALID_ARG;
    if (head_dim < 8 || head_dim > 256 || head_dim % 8) return H3QK_ERR_INVALID_ARG;
    if (rotary_dim < 0 || rotary_dim > head_dim || rotary_dim % 2) return H3QK_ERR_INVALID_ARG;
    if (o.batch < 1 || tokens % o.batch) return H3QK_ERR_INVALID_ARG;
    const int64_t S = tokens / o.batch;
    if (valid_len < 0 || valid_len > S) return H3QK_ERR_INVALID_ARG;
    if (o.n_axes != 1 && o.n_axes != 3) return H3QK_ERR_INVALID_ARG;
    int dims[3] = {o.axis_dims[0], o.axis_dims[1], o.axis_dims[2]};
    if (dims[0] == 0 && dims[1] == 0 && dims[2] == 0) {
        if (o.n_axes == 3) {
            if (rotary_dim % 3) return H3QK_ERR_INVALID_ARG;
            dims[0] = dims[1] = dims[2] = rotary_dim / 3;
        } else {
            dims[0] = rotary_dim;
        }
    }
    int dim_sum = 0;
    for (int a = 0; a < 3; ++a) {
        if (a >= o.n_axes && dims[a] != 0) return H3QK_ERR_INVALID_ARG;
        if (dims[a] < 0 || dims[a] % 2) return H3QK_ERR_INVALID_ARG;
        dim_sum += dims[a];
    }
    if (dim_sum != rotary_dim) return H3QK_ERR_INVALID_ARG;
    if (!(o.eps >= 0.0f) || !std::isfinite(o.eps)) return H3QK_ERR_INVALID_ARG;
    if (!(o.theta > 0.0) || !std::isfinite(o.theta)) return H3QK_ERR_INVALID_ARG;
    int in_dtype = o.in_dtype == H3QK_DTYPE_DEFAULT ? default_in : o.in_dtype;
    if (in_dtype != H3QK_FP16 && in_dtype != H3QK_BF16) return H3QK_ERR_INVALID_ARG;

    const int64_t HD = static_cast<int64_t>(heads) * head_dim;
    const int64_t stride = o.qkv_row_stride ? o.qkv_row_stride : parts * HD;
    if (stride < parts * HD) return H3QK_ERR_INVALID_ARG;
    // Byte sizes must stay far from int64 overflow.
    if (tokens > 0 && (stride > (INT64_C(1) << 40) / tokens || HD > (INT64_C(1) << 40) / tokens))
        return H3QK_ERR_INVALID_ARG;
    if (o.out_layout != H3QK_LAYOUT_HEAD_MAJOR && o.out_layout != H3QK_LAYOUT_TOKEN_MAJOR)
        return H3QK_ERR_INVALID_ARG;

    // An empty call (tokens == 0) reads and writes no row, so its row buffers
    // may be NULL (an empty torch tensor has a null data pointer).
    if (!norm_wq || !norm_wk) return H3QK_ERR_INVALID_ARG;
    if (tokens > 0 && !qkv) return H3QK_ERR_INVALID_ARG;
    if (tokens > 0 && rotary_dim > 0 && !positions) return H3QK_ERR_INVALID_ARG;
    if (stride % 8) return H3QK_ERR_MISALIGNED;
    if (!aligned(qkv, 16) || !aligned(norm_wq, 16) || !aligned(norm_wk, 16)) return H3QK_ERR_MISALIGNED;
    if (positions && !aligned(positions, 4)) return H3QK_ERR_MISALIGNED;
    if (o.valid_lens && !aligned(o.valid_lens, 4)) return H3QK_ERR_MISALIGNED;
    if (o.sat_counts && !aligned(o.sat_counts, 4)) return H3QK_ERR_MISALIGNED;

    plan->ins[0] = range_of(qkv, tokens > 0 ? ((tokens - 1) * stride + parts * HD) * 2 : 0);
    plan->ins[1] = range_of(norm_wq, head_dim * 4);
    plan->ins[2] = range_of(norm_wk, head_dim * 4);
    plan->ins[3] = range_of(positions, positions ? tokens * o.n_axes * 4 : 0);
    plan->ins[4] = range_of(o.valid_lens, o.valid_lens ? o.batch * 4 : 0);
    plan->HD = HD;

    h3qk::Params& p = plan->p;
    std::memset(&p, 0, sizeof(p));
    p.qkv = static_cast<const uint16_t*>(qkv);
    p.wq = norm_wq;
    p.wk = norm_wk;
    p.pos = positions;
    p.rows = tokens;
    p.seq = S;
    p.valid_len = valid_len;
    p.row_stride = stride;
    p.heads = heads;
    p.head_dim = head_dim;
    p.rotary_dim = rotary_dim;
    p.n_axes = o.n_axes;
    p.chunks = head_dim / 8;
    p.eps = o.eps;
    p.inv_d = (head_dim & (head_dim - 1)) == 0 ? 1.0f / static_cast<float>(head_dim) : 0.0f;
    p.one2 = make_float2(1.0f, 1.0f);
    p.mone2 = make_float2(-1.0f, -1.0f);
    // Packed rows [Q | K | V]; all three parts; one slot per part.
    p.in_part_off[0] = 0;
    p.in_part_off[1] = HD;
    p.in_part_off[2] = 2 * HD;
    p.pf_span = parts * HD;
    p.dbg_status = dbg_status_addr();
    p.dbg_out_elems = tokens * HD;
    {
        std::lock_guard<std::mutex> lock(g_dbg_mu);
        if (g_dbg_out_limit >= 0 && g_dbg_out_limit < p.dbg_out_elems) p.dbg_out_elems = g_dbg_out_limit;
    }
    p.qk_first = 0;
    p.qk_end = 2;
    p.has_v = 1;
    p.slot[0] = 0;
    p.slot[1] = 1;
    p.slot[2] = 2;
    p.valid_lens = o.valid_lens;
    if (o.out_layout == H3QK_LAYOUT_TOKEN_MAJOR) {
        p.out_bstride = S * HD;
        p.out_sstride = HD;
        p.out_hstride = head_dim;
    } else {
        p.out_bstride = static_cast<int64_t>(heads) * S * head_dim;
        p.out_sstride = head_dim;
        p.out_hstride = S * head_dim;
    }
    // Rotary inverse frequencies theta^(-2i/d_a), in double, rounded once.
    int pair = 0;
    for (int a = 0; a < o.n_axes; ++a)
        for (int i = 0; i < dims[a] / 2; ++i, ++pair) {
            const double expo = -(2.0 * static_cast<double>(i)) / static_cast<double>(dims[a]);
            p.inv_freq[pair] = static_cast<float>(std::pow(o.theta, expo));
            p.axis[pair] = static_cast<uint8_t>(a);
        }

    plan->P = next_pow2(head_dim / 8);
    plan->st = reinterpret_cast<cudaStream_t>(stream);
    plan->bf16 = in_dtype == H3QK_BF16;
    return H3QK_OK;
}

// True when range r overlaps any input of the plan.
bool overlaps_inputs(const Plan& pl, Range r)
{
    for (int k = 0; k < 5; ++k)
        if (overlap(r, pl.ins[k])) return true;
    return false;
}

// The buffers a call writes besides its outputs (the amax workspace, zeroed
// on the stream before the amax pass, and the saturation counters) must not
// overlap an input, the static table or each other.  extra = {static table,
// workspace, counters}, each an empty range when the call does not use it.
bool scratch_overlaps(const Plan& pl, const Range (&extra)[3])
{
    for (int k = 1; k < 3; ++k) {
        if (overlaps_inputs(pl, extra[k])) return true;
        if (overlap(extra[k], extra[0])) return true;
    }
    return overlap(extra[1], extra[2]);
}

// Zero the amax words, then run the amax pass (skipped when no row is valid).
cudaError_t launch_amax_init(unsigned int* words, cudaStream_t st)
{
    h3qk::amax_init_kernel<<<1, 32, 0, st>>>(words);
    ++g_launches;
    return cudaGetLastError();
}

h3qk_status run_amax(const Plan& pl)
{
    h3qk::amax_init_kernel<<<1, 32, 0, pl.st>>>(pl.p.amax_words);
    ++g_launches;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    if (pl.p.rows > 0 && (pl.p.valid_len > 0 || pl.p.valid_lens)) {
        h3qk::Params pa = pl.p;
        pa.chained = 1;  // a programmatic dependent of the zeroing kernel
        e = launch(pl.bf16, pl.P, h3qk::kAmax, pa, pl.st);
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return H3QK_OK;
}

}  // namespace h3qk_detail

using namespace h3qk_detail;


extern "C" {

h3qk_status h3qk_prepare(const void* qkv, const float* norm_wq, const float* norm_wk,
                         const int32_t* positions, int64_t tokens, int32_t heads,
                         int32_t head_dim, int32_t rotary_dim, int64_t valid_len,
                         h3qk_dtype out_dtype, h3qk_scale_mode scale_mode, void* out_q,
                         void* out_k, void* out_v, float* out_scales, const h3qk_opts* opts,
                         h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    const bool e4m3 = out_dtype == H3QK_E4M3;
    Plan pl;
    h3qk_status s = plan_inputs(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                                valid_len, out_dtype == H3QK_FP16 ? H3QK_FP16 : H3QK_BF16, o, stream, &pl);
    if (s != H3QK_OK) return s;
    const int in_dtype = pl.bf16 ? H3QK_BF16 : H3QK_FP16;
    if (out_dtype == H3QK_FP16 || out_dtype == H3QK_BF16) {
        if (out_dtype != in_dtype || scale_mode != H3QK_SCALE_NONE) return H3QK_ERR_INVALID_ARG;
    } else if (e4m3) {
        if (scale_mode != H3QK_SCALE_DYNAMIC && scale_mode != H3QK_SCALE_STATIC) return H3QK_ERR_INVALID_ARG;
    } else {
        return H3QK_ERR_INVALID_ARG;
    }
    if (tokens > 0 && (!out_q || !out_k || !out_v)) return H3QK_ERR_INVALID_ARG;
    if (e4m3 && !out_scales) return H3QK_ERR_INVALID_ARG;
    if (e4m3 && scale_mode == H3QK_SCALE_STATIC && !o.static_scales) return H3QK_ERR_INVALID_ARG;
    if (e4m3 && scale_mode == H3QK_SCALE_DYNAMIC &&
        (!o.workspace || o.workspace_bytes < h3qk_workspace_bytes()))
        return H3QK_ERR_INVALID_ARG;
    if (!aligned(out_q, 16) || !aligned(out_k, 16) || !aligned(out_v, 16)) return H3QK_ERR_MISALIGNED;
    if (e4m3 && !aligned(out_scales, 4)) return H3QK_ERR_MISALIGNED;
    if (e4m3 && scale_mode == H3QK_SCALE_STATIC && !aligned(o.static_scales, 4)) return H3QK_ERR_MISALIGNED;
    if (e4m3 && scale_mode == H3QK_SCALE_DYNAMIC && !aligned(o.workspace, 16)) return H3QK_ERR_MISALIGNED;

    // Aliasing: outputs never overlap inputs or each other.
    const int64_t esz = e4m3 ? 1 : 2;
    const int64_t n_out = tokens * pl.HD * esz;
    const Range outs[4] = {range_of(out_q, n_out), range_of(out_k, n_out), range_of(out_v, n_out),
                           range_of(out_scales, e4m3 ? 12 : 0)};
    const Range extra[3] = {
        range_of(o.static_scales, (e4m3 && scale_mode == H3QK_SCALE_STATIC) ? 12 : 0),
        range_of(o.workspace, (e4m3 && scale_mode == H3QK_SCALE_DYNAMIC) ? 16 : 0),
        range_of(o.sat_counts, (e4m3 && o.sat_counts) ? 12 : 0)};
    for (int i = 0; i < 4; ++i) {
        for (int k = i + 1; k < 4; ++k)
            if (overlap(outs[i], outs[k])) return H3QK_ERR_ALIAS;
        if (overlaps_inputs(pl, outs[i])) return H3QK_ERR_ALIAS;
        for (int k = 0; k < 3; ++k)
            if (overlap(outs[i], extra[k])) return H3QK_ERR_ALIAS;
    }
    if (scratch_overlaps(pl, extra)) return H3QK_ERR_ALIAS;

    h3qk::Params& p = pl.p;
    p.out[0] = out_q;
    p.out[1] = out_k;
    p.out[2] = out_v;
    p.out_scales = out_scales;
    p.amax_words = static_cast<unsigned int*>(o.workspace);
    p.scale_words = scale_mode == H3QK_SCALE_DYNAMIC
                        ? p.amax_words
                        : reinterpret_cast<const unsigned int*>(o.static_scales);
    p.dynamic = scale_mode == H3QK_SCALE_DYNAMIC ? 1 : 0;
    p.sat_counts = e4m3 ? o.sat_counts : nullptr;
    cudaError_t e;
    if (!e4m3) {
        if (tokens == 0 || (valid_len == 0 && !o.valid_lens)) return H3QK_OK;
        e = launch(pl.bf16, pl.P, h3qk::kOut16, p, pl.st);
        return e == cudaSuccess ? H3QK_OK : fail_cuda(e);
    }
    if (scale_mode == H3QK_SCALE_DYNAMIC) {
        s = run_amax(pl);
        if (s != H3QK_OK) return s;
        p.chained = 1;  // a programmatic dependent of the amax pass
        p.reverse = 1;  // starts with the rows the amax pass read last (in L2)
    }
    e = launch(pl.bf16, pl.P, h3qk::kCast, p, pl.st);
    return e == cudaSuccess ? H3QK_OK : fail_cuda(e);
}

h3qk_status h3qk_amax(const void* qkv, const float* norm_wq, const float* norm_wk,
                      const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                      int32_t rotary_dim, int64_t valid_len, float* out_amax, const h3qk_opts* opts,
                      h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    Plan pl;
    h3qk_status s = plan_inputs(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                                valid_len, H3QK_BF16, o, stream, &pl);
    if (s != H3QK_OK) return s;
    if (!out_amax) return H3QK_ERR_INVALID_ARG;
    if (!aligned(out_amax, 4)) return H3QK_ERR_MISALIGNED;
    if (overlaps_inputs(pl, range_of(out_amax, 12))) return H3QK_ERR_ALIAS;
    pl.p.amax_words = reinterpret_cast<unsigned int*>(out_amax);
    return run_amax(pl);
}

h3qk_status h3qk_norm_rope_tensor(const void* x, const float* norm_w, const int32_t* positions,
                                  int64_t tokens, int32_t heads, int32_t head_dim,
                                  int32_t rotary_dim, int64_t valid_len, h3qk_tensor_kind kind,
                                  h3qk_dtype out_dtype, h3qk_scale_mode scale_mode, void* out,
                                  float* out_scale, const h3qk_opts* opts, h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    if (kind != H3QK_TENSOR_Q && kind != H3QK_TENSOR_K && kind != H3QK_TENSOR_V) return H3QK_ERR_INVALID_ARG;
    // V needs no weight; its weight pointers are a stand-in that no kernel reads.
    alignas(16) static const float kNoWeight[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float* w = norm_w ? norm_w : (kind == H3QK_TENSOR_V ? kNoWeight : nullptr);
    o.out_layout = H3QK_LAYOUT_TOKEN_MAJOR;
    const bool e4m3 = out_dtype == H3QK_E4M3;
    Plan pl;
    h3qk_status s = plan_inputs(x, w, w, positions, tokens, heads, head_dim, rotary_dim, valid_len,
                                out_dtype == H3QK_FP16 ? H3QK_FP16 : H3QK_BF16, o, stream, &pl, 1);
    if (s != H3QK_OK) return s;
    if (kind == H3QK_TENSOR_V) pl.ins[1] = pl.ins[2] = Range{0, 0};
    const int in_dtype = pl.bf16 ? H3QK_BF16 : H3QK_FP16;
    if (out_dtype == H3QK_FP16 || out_dtype == H3QK_BF16) {
        if (out_dtype != in_dtype || scale_mode != H3QK_SCALE_NONE) return H3QK_ERR_INVALID_ARG;
    } else if (e4m3) {
        if (scale_mode != H3QK_SCALE_DYNAMIC && scale_mode != H3QK_SCALE_STATIC) return H3QK_ERR_INVALID_ARG;
    } else {
        return H3QK_ERR_INVALID_ARG;
    }
    if (tokens > 0 && !out) return H3QK_ERR_INVALID_ARG;
    if (e4m3 && !out_scale) return H3QK_ERR_INVALID_ARG;
    if (e4m3 && scale_mode == H3QK_SCALE_STATIC && !o.static_scales) return H3QK_ERR_INVALID_ARG;
    if (e4m3 && scale_mode == H3QK_SCALE_DYNAMIC &&
        (!o.workspace || o.workspace_bytes < h3qk_workspace_bytes()))
        return H3QK_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return H3QK_ERR_MISALIGNED;
    if (e4m3 && !aligned(out_scale, 4)) return H3QK_ERR_MISALIGNED;
    if (e4m3 && scale_mode == H3QK_SCALE_STATIC && !aligned(o.static_scales, 4)) return H3QK_ERR_MISALIGNED;
    if (e4m3 && scale_mode == H3QK_SCALE_DYNAMIC && !aligned(o.workspace, 16)) return H3QK_ERR_MISALIGNED;
    const Range ro = range_of(out, tokens * pl.HD * (e4m3 ? 1 : 2));
    const Range rs = range_of(out_scale, e4m3 ? 4 : 0);
    const Range extra[3] = {
        range_of(o.static_scales, (e4m3 && scale_mode == H3QK_SCALE_STATIC) ? 4 : 0),
        range_of(o.workspace, (e4m3 && scale_mode == H3QK_SCALE_DYNAMIC) ? 16 : 0),
        range_of(o.sat_counts, (e4m3 && o.sat_counts) ? 4 : 0)};
    if (overlap(ro, rs) || overlaps_inputs(pl, ro) || overlaps_inputs(pl, rs)) return H3QK_ERR_ALIAS;
    for (int k = 0; k < 3; ++k)
        if (overlap(ro, extra[k]) || overlap(rs, extra[k])) return H3QK_ERR_ALIAS;
    if (scratch_overlaps(pl, extra)) return H3QK_ERR_ALIAS;

    h3qk::Params& p = pl.p;
    const int t = static_cast<int>(kind);
    p.in_part_off[0] = p.in_part_off[1] = p.in_part_off[2] = 0;
    p.qk_first = t < 2 ? t : 0;
    p.qk_end = t < 2 ? t + 1 : 0;
    p.has_v = t == 2 ? 1 : 0;
    p.slot[0] = p.slot[1] = p.slot[2] = -1;
    p.slot[t] = 0;
    p.out[0] = p.out[1] = p.out[2] = out;
    p.out_scales = out_scale;
    p.amax_words = static_cast<unsigned int*>(o.workspace);
    p.scale_words = scale_mode == H3QK_SCALE_DYNAMIC
                        ? p.amax_words
                        : reinterpret_cast<const unsigned int*>(o.static_scales);
    p.dynamic = scale_mode == H3QK_SCALE_DYNAMIC ? 1 : 0;
    p.sat_counts = e4m3 ? o.sat_counts : nullptr;
    cudaError_t e;
    if (!e4m3) {
        if (tokens == 0 || (valid_len == 0 && !o.valid_lens)) return H3QK_OK;
        e = launch(pl.bf16, pl.P, h3qk::kOut16, p, pl.st);
        return e == cudaSuccess ? H3QK_OK : fail_cuda(e);
    }
    if (scale_mode == H3QK_SCALE_DYNAMIC) {
        s = run_amax(pl);
        if (s != H3QK_OK) return s;
        p.chained = 1;  // a programmatic dependent of the amax pass
        p.reverse = 1;  // starts with the rows the amax pass read last (in L2)
    }
    e = launch(pl.bf16, pl.P, h3qk::kCast, p, pl.st);
    return e == cudaSuccess ? H3QK_OK : fail_cuda(e);
}

h3qk_status h3qk_cast(const void* qkv, const float* norm_wq, const float* norm_wk,
                      const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                      int32_t rotary_dim, int64_t valid_len, const float* amax, void* out_q,
                      void* out_k, void* out_v, float* out_scales, const h3qk_opts* opts,
                      h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    Plan pl;
    h3qk_status s = plan_inputs(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                                valid_len, H3QK_BF16, o, stream, &pl);
    if (s != H3QK_OK) return s;
    if (!amax || !out_scales) return H3QK_ERR_INVALID_ARG;
    if (tokens > 0 && (!out_q || !out_k || !out_v)) return H3QK_ERR_INVALID_ARG;
    if (!aligned(amax, 4) || !aligned(out_scales, 4)) return H3QK_ERR_MISALIGNED;
    if (!aligned(out_q, 16) || !aligned(out_k, 16) || !aligned(out_v, 16)) return H3QK_ERR_MISALIGNED;
    const int64_t n_out = tokens * pl.HD;
    const Range outs[4] = {range_of(out_q, n_out), range_of(out_k, n_out), range_of(out_v, n_out),
                           range_of(out_scales, 12)};
    const Range amax_r = range_of(amax, 12);
    for (int i = 0; i < 4; ++i) {
        for (int k = i + 1; k < 4; ++k)
            if (overlap(outs[i], outs[k])) return H3QK_ERR_ALIAS;
        if (overlaps_inputs(pl, outs[i]) || overlap(outs[i], amax_r)) return H3QK_ERR_ALIAS;
    }
    h3qk::Params& p = pl.p;
    p.out[0] = out_q;
    p.out[1] = out_k;
    p.out[2] = out_v;
    p.out_scales = out_scales;
    p.scale_words = reinterpret_cast<const unsigned int*>(amax);
    p.dynamic = 1;
    if (o.sat_counts) {
        if (overlaps_inputs(pl, range_of(o.sat_counts, 12)) || overlap(range_of(o.sat_counts, 12), amax_r))
            return H3QK_ERR_ALIAS;
        for (int i = 0; i < 4; ++i)
            if (overlap(outs[i], range_of(o.sat_counts, 12))) return H3QK_ERR_ALIAS;
        p.sat_counts = o.sat_counts;
    }
    const cudaError_t e = launch(pl.bf16, pl.P, h3qk::kCast, p, pl.st);
    return e == cudaSuccess ? H3QK_OK : fail_cuda(e);
}

h3qk_status h3qk_prepare_sage(const void* qkv, const float* norm_wq, const float* norm_wk,
                              const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                              int32_t rotary_dim, int64_t valid_len, float kv_scale, float* out_q,
                              float* out_k, void* out_v, const h3qk_opts* opts, h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    Plan pl;
    h3qk_status s = plan_inputs(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                                valid_len, H3QK_BF16, o, stream, &pl);
    if (s != H3QK_OK) return s;
    if (!std::isfinite(kv_scale)) return H3QK_ERR_INVALID_ARG;
    if (tokens > 0 && (!out_q || !out_k || !out_v)) return H3QK_ERR_INVALID_ARG;
    if (!aligned(out_q, 16) || !aligned(out_k, 16) || !aligned(out_v, 16)) return H3QK_ERR_MISALIGNED;
    const Range outs[3] = {range_of(out_q, tokens * pl.HD * 4), range_of(out_k, tokens * pl.HD * 4),
                           range_of(out_v, tokens * pl.HD * 2)};
    for (int i = 0; i < 3; ++i) {
        for (int k = i + 1; k < 3; ++k)
            if (overlap(outs[i], outs[k])) return H3QK_ERR_ALIAS;
        if (overlaps_inputs(pl, outs[i])) return H3QK_ERR_ALIAS;
    }
    h3qk::Params& p = pl.p;
    p.out[0] = out_q;
    p.out[1] = out_k;
    p.out[2] = out_v;
    p.kv_scale = kv_scale;
    if (tokens == 0 || (valid_len == 0 && !o.valid_lens)) return H3QK_OK;
    const cudaError_t e = launch(pl.bf16, pl.P, h3qk::kSage, p, pl.st);
    return e == cudaSuccess ? H3QK_OK : fail_cuda(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// h3qk_prepare_noalloc: h3qk_prepare for callers that cannot allocate device
// memory.  Its only scratch is the fixed array below (the three amax words of
// a DYNAMIC call); every GPU that loads this library holds it until exit.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoallocScratchBytes = 256;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoallocScratchBytes / 4];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in for the device array).
h3qk_status noalloc_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return H3QK_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return fail_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return H3QK_OK;
}

}  // namespace

extern "C" h3qk_status h3qk_prepare_noalloc(const void* qkv, const float* norm_wq,
                                            const float* norm_wk, const int32_t* positions,
                                            int64_t tokens, int32_t heads, int32_t head_dim,
                                            int32_t rotary_dim, int64_t valid_len,
                                            h3qk_dtype out_dtype, h3qk_scale_mode scale_mode,
                                            void* out_q, void* out_k, void* out_v,
                                            float* out_scales, const h3qk_opts* opts,
                                            h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    if (scale_mode == H3QK_SCALE_DYNAMIC) {
        // The scratch a call needs must fit the fixed array.  A DYNAMIC call
        // needs h3qk_workspace_bytes() = 16 bytes whatever its sizes, so this
        // rejects nothing today; it keeps the limit explicit.
        if (h3qk_workspace_bytes() > kNoallocScratchBytes) return H3QK_ERR_INVALID_ARG;
        void* ws = nullptr;
        const h3qk_status st = noalloc_scratch(&ws);
        if (st != H3QK_OK) return st;
        // The kernels clear the amax words at the start of every DYNAMIC call.
        o.workspace = ws;
        o.workspace_bytes = kNoallocScratchBytes;
    }
    return h3qk_prepare(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                        valid_len, out_dtype, scale_mode, out_q, out_k, out_v, out_scales, &o,
                        stream);
}
