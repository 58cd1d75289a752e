#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "h3qk.h"
#include "h3qk_internal.h"

using namespace h3qk_detail;

// h3qk_prepare_host: the path on host buffers.  The call is cut into chunks
// of about H3QK_HOST_CHUNK_BYTES of input rows (chunk_rows below) inside one
// item; three streams of the
// library (host -> device copies, kernels, device -> host copies) keep the
// copies of one chunk in flight while another computes.  Device memory comes
// from the caller's workspace: a ring of kHostSlots chunk slots (or, for
// dynamic e4m3, the whole input, which the cast pass reads after the amax
// pass has seen every row).
namespace {

constexpr int kMaxDevices = 64;
constexpr int kHostSlots = 3;

// Input bytes per chunk.  Smaller chunks shorten the pipeline's fill (the
// first chunk's copy in) and drain (the last chunk's copy out), larger ones
// pay the per-copy cost less often.  On the 65k tile's two calls (GB300) the
// step took 17.7 ms at 8,192-row chunks (151 MB), 17.3 ms at 64 MiB, 17.9 ms
// at 32 MiB, 18.3 ms at 16 MiB and 19.8 ms at 8 MiB.
#ifndef H3QK_HOST_CHUNK_BYTES
#define H3QK_HOST_CHUNK_BYTES (64 << 20)
#endif

// Rows per chunk: H3QK_HOST_CHUNK_BYTES of input rows, between 256 and
// 8,192 rows, never more than the rows of one item.
int64_t chunk_rows(int64_t seq, int64_t stride)
{
    int64_t n = static_cast<int64_t>(H3QK_HOST_CHUNK_BYTES) / (stride * 2);
    n = n < 256 ? 256 : (n > 8192 ? 8192 : n);
    return seq < n ? seq : n;
}

struct HostStreams {
    std::mutex call;                                   // one host call enqueues at a time
    cudaStream_t s[3] = {nullptr, nullptr, nullptr};  // h2d, compute, d2h
    cudaEvent_t in[kHostSlots] = {};                   // chunk copied in
    cudaEvent_t cmp[kHostSlots] = {};                  // chunk computed
    cudaEvent_t out[kHostSlots] = {};                  // chunk copied out
    cudaEvent_t start = nullptr, done = nullptr, last = nullptr;
    bool ready = false;
};
std::mutex g_host_mu;
HostStreams g_host[kMaxDevices];

// The library's streams and events of the current device, created on first use.
h3qk_status host_streams(HostStreams** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return h3qk_internal_fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return H3QK_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostStreams& h = g_host[dev];
    if (!h.ready) {
        // A handle made by an earlier, failed attempt is kept and not made
        // again, so a retry after a failure leaks nothing.
        for (auto& st : h.s)
            if (!st && (e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking)) != cudaSuccess) {
                st = nullptr;
                return h3qk_internal_fail_cuda(e);
            }
        auto make_event = [&](cudaEvent_t* ev) {
            if (*ev) return cudaSuccess;
            const cudaError_t r = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
            if (r != cudaSuccess) *ev = nullptr;
            return r;
        };
        for (cudaEvent_t* ev : {&h.start, &h.done, &h.last})
            if ((e = make_event(ev)) != cudaSuccess) return h3qk_internal_fail_cuda(e);
        for (int k = 0; k < kHostSlots; ++k)
            for (cudaEvent_t* ev : {&h.in[k], &h.cmp[k], &h.out[k]})
                if ((e = make_event(ev)) != cudaSuccess) return h3qk_internal_fail_cuda(e);
        h.ready = true;
    }
    *out = &h;
    return H3QK_OK;
}

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Byte offsets of the parts of the host-call workspace.
struct HostLayout {
    size_t w = 0, misc = 0, in = 0, pos = 0, out = 0, total = 0;
    size_t in_slot = 0, pos_slot = 0;  // bytes per input slot (dynamic: the whole input)
    size_t out_t = 0, out_slot = 0;    // bytes per output tensor of a slot, per slot
    int64_t chunk = 0;
};

HostLayout host_layout(int64_t tokens, int64_t seq, int32_t heads, int32_t head_dim, int64_t stride, int32_t n_axes,
                       bool e4m3, bool dynamic)
{
    HostLayout L;
    const int64_t HD = static_cast<int64_t>(heads) * head_dim;
    L.chunk = chunk_rows(seq, stride);
    size_t off = 0;
    L.w = off;
    off += round256(2 * static_cast<size_t>(head_dim) * 4);
    L.misc = off;  // static table (3 floats), amax words (4), descales (3)
    off += 256;
    const size_t rows_in = dynamic ? static_cast<size_t>(tokens) : static_cast<size_t>(L.chunk);
    L.in_slot = round256(rows_in * static_cast<size_t>(stride) * 2);
    L.pos_slot = round256(rows_in * static_cast<size_t>(n_axes) * 4);
    const int in_slots = dynamic ? 1 : kHostSlots;
    L.in = off;
    off += in_slots * L.in_slot;
    L.pos = off;
    off += in_slots * L.pos_slot;
    L.out_t = round256(static_cast<size_t>(L.chunk) * HD * (e4m3 ? 1 : 2));
    L.out_slot = 3 * L.out_t;
    L.out = off;
    off += kHostSlots * L.out_slot;
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

size_t h3qk_host_workspace_bytes(int64_t tokens, int32_t heads, int32_t head_dim, h3qk_dtype out_dtype,
                                 h3qk_scale_mode scale_mode, const h3qk_opts* opts)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    if (tokens < 0 || heads < 1 || head_dim < 8 || o.batch < 1 || tokens % o.batch) return 0;
    const int64_t HD = static_cast<int64_t>(heads) * head_dim;
    const int64_t stride = o.qkv_row_stride ? o.qkv_row_stride : 3 * HD;
    const bool e4m3 = out_dtype == H3QK_E4M3;
    return host_layout(tokens, tokens / o.batch, heads, head_dim, stride, o.n_axes, e4m3,
                       e4m3 && scale_mode == H3QK_SCALE_DYNAMIC)
        .total;
}

h3qk_status h3qk_prepare_host(const void* qkv, const float* norm_wq, const float* norm_wk,
                              const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                              int32_t rotary_dim, int64_t valid_len, h3qk_dtype out_dtype,
                              h3qk_scale_mode scale_mode, void* out_q, void* out_k, void* out_v,
                              float* out_scales, const h3qk_opts* opts, void* workspace,
                              size_t workspace_bytes, h3qk_stream_t stream)
{
    h3qk_opts o;
    h3qk_opts_init(&o);
    if (opts) o = *opts;
    const bool e4m3 = out_dtype == H3QK_E4M3;
    const bool dynamic = e4m3 && scale_mode == H3QK_SCALE_DYNAMIC;
    // Host-side checks of the whole call: the sizes and options through the
    // device entry's validator, with the (aligned) workspace standing in for
    // every device pointer; nothing is dereferenced here.
    if (!workspace || !aligned(workspace, 256)) return workspace ? H3QK_ERR_MISALIGNED : H3QK_ERR_INVALID_ARG;
    if (o.sat_counts || o.workspace) return H3QK_ERR_INVALID_ARG;  // not part of this entry
    if (!norm_wq || !norm_wk) return H3QK_ERR_INVALID_ARG;
    h3qk_opts ov = o;
    ov.valid_lens = nullptr;
    Plan whole;
    h3qk_status s = plan_inputs(workspace, static_cast<const float*>(workspace), static_cast<const float*>(workspace),
                                rotary_dim > 0 ? static_cast<const int32_t*>(workspace) : nullptr, tokens, heads,
                                head_dim, rotary_dim, valid_len,
                                out_dtype == H3QK_FP16 ? H3QK_FP16 : H3QK_BF16, ov, stream, &whole);
    if (s != H3QK_OK) return s;
    const int in_dtype = whole.bf16 ? H3QK_BF16 : H3QK_FP16;
    if (out_dtype == H3QK_FP16 || out_dtype == H3QK_BF16) {
        if (out_dtype != in_dtype || scale_mode != H3QK_SCALE_NONE) return H3QK_ERR_INVALID_ARG;
    } else if (e4m3) {
        if (scale_mode != H3QK_SCALE_DYNAMIC && scale_mode != H3QK_SCALE_STATIC) return H3QK_ERR_INVALID_ARG;
        if (!out_scales) return H3QK_ERR_INVALID_ARG;
        if (scale_mode == H3QK_SCALE_STATIC && !o.static_scales) return H3QK_ERR_INVALID_ARG;
    } else {
        return H3QK_ERR_INVALID_ARG;
    }
    if (tokens > 0 && (!qkv || !out_q || !out_k || !out_v)) return H3QK_ERR_INVALID_ARG;
    if (tokens > 0 && rotary_dim > 0 && !positions) return H3QK_ERR_INVALID_ARG;
    const int64_t B = o.batch, S = tokens / o.batch, HD = whole.HD, D = head_dim;
    const int64_t stride = whole.p.row_stride;
    const int64_t esz = e4m3 ? 1 : 2;
    const HostLayout L = host_layout(tokens, S, heads, head_dim, stride, o.n_axes, e4m3, dynamic);
    if (workspace_bytes < L.total) return H3QK_ERR_INVALID_ARG;

    HostStreams* hs = nullptr;
    if ((s = host_streams(&hs)) != H3QK_OK) return s;
    std::lock_guard<std::mutex> call_lock(hs->call);
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t h2d = hs->s[0], cmp = hs->s[1], d2h = hs->s[2];
    char* ws = static_cast<char*>(workspace);
    float* w_dev = reinterpret_cast<float*>(ws + L.w);
    float* table_dev = reinterpret_cast<float*>(ws + L.misc);
    unsigned int* amax_dev = reinterpret_cast<unsigned int*>(ws + L.misc + 64);
    float* scales_dev = reinterpret_cast<float*>(ws + L.misc + 128);
    cudaError_t e;
#define H3QK_TRY(x)                               \
    do {                                          \
        if ((e = (x)) != cudaSuccess) return h3qk_internal_fail_cuda(e); \
    } while (0)

    // Start after the caller's earlier work on its stream.
    H3QK_TRY(cudaEventRecord(hs->start, caller));
    for (cudaStream_t st : {h2d, cmp, d2h}) H3QK_TRY(cudaStreamWaitEvent(st, hs->start, 0));
    H3QK_TRY(cudaMemcpyAsync(w_dev, norm_wq, D * 4, cudaMemcpyHostToDevice, h2d));
    H3QK_TRY(cudaMemcpyAsync(w_dev + D, norm_wk, D * 4, cudaMemcpyHostToDevice, h2d));
    if (e4m3 && !dynamic) H3QK_TRY(cudaMemcpyAsync(table_dev, o.static_scales, 12, cudaMemcpyHostToDevice, h2d));
    H3QK_TRY(cudaEventRecord(hs->last, h2d));
    H3QK_TRY(cudaStreamWaitEvent(cmp, hs->last, 0));

    // Per-chunk device call options: one item of the chunk's valid rows.
    h3qk_opts oc = o;
    oc.batch = 1;
    oc.valid_lens = nullptr;
    oc.sat_counts = nullptr;
    oc.static_scales = table_dev;
    oc.workspace = amax_dev;
    oc.workspace_bytes = 16;
    const bool token_major = o.out_layout == H3QK_LAYOUT_TOKEN_MAJOR;

    // Copy the n valid rows of chunk (item b, first row a) into input slot `si`.
    auto copy_in = [&](int64_t b, int64_t a, int64_t n, int si) -> cudaError_t {
        const int64_t r0 = b * S + a;
        char* dst = ws + L.in + si * L.in_slot;
        const size_t bytes = static_cast<size_t>((n - 1) * stride + 3 * HD) * 2;
        cudaError_t ee = cudaMemcpyAsync(dst, static_cast<const uint16_t*>(qkv) + r0 * stride, bytes,
                                         cudaMemcpyHostToDevice, h2d);
        if (ee != cudaSuccess || !positions) return ee;
        return cudaMemcpyAsync(ws + L.pos + si * L.pos_slot, positions + r0 * o.n_axes, n * o.n_axes * 4,
                               cudaMemcpyHostToDevice, h2d);
    };
    // Copy the n valid output rows of output slot `so` to the host tensors.
    auto copy_out = [&](int64_t b, int64_t a, int64_t n, int so) -> cudaError_t {
        void* hosts[3] = {out_q, out_k, out_v};
        for (int t = 0; t < 3; ++t) {
            const char* src = ws + L.out + so * L.out_slot + t * L.out_t;
            char* dst = static_cast<char*>(hosts[t]);
            cudaError_t ee;
            if (token_major) {
                ee = cudaMemcpyAsync(dst + (b * S + a) * HD * esz, src, n * HD * esz, cudaMemcpyDeviceToHost, d2h);
            } else {
                ee = cudaMemcpy2DAsync(dst + ((b * heads) * S + a) * D * esz, S * D * esz, src, n * D * esz,
                                       n * D * esz, heads, cudaMemcpyDeviceToHost, d2h);
            }
            if (ee != cudaSuccess) return ee;
        }
        return cudaSuccess;
    };
    auto out_ptr = [&](int so, int t) -> void* {
        return ws + L.out + so * L.out_slot + t * L.out_t;
    };

    // The chunks that hold valid rows.
    struct Chunk {
        int64_t b, a, n;
    };
    std::vector<Chunk> chunks;
    for (int64_t b = 0; b < B; ++b) {
        int64_t vl = valid_len;
        if (o.valid_lens) {
            vl = o.valid_lens[b];  // host array
            vl = vl < 0 ? 0 : (vl > S ? S : vl);
        }
        for (int64_t a = 0; a < vl; a += L.chunk) chunks.push_back({b, a, (vl - a) < L.chunk ? (vl - a) : L.chunk});
    }
    const int64_t n_chunks = static_cast<int64_t>(chunks.size());

    if (dynamic) {
        H3QK_TRY(launch_amax_init(amax_dev, cmp));
        // Pass 1: every chunk into the resident input, its rows into the amax.
        int64_t row_off = 0;
        std::vector<int64_t> offs(n_chunks);
        for (int64_t k = 0; k < n_chunks; ++k) {
            const Chunk& c = chunks[k];
            offs[k] = row_off;
            const int64_t r0 = c.b * S + c.a;
            const size_t bytes = static_cast<size_t>((c.n - 1) * stride + 3 * HD) * 2;
            H3QK_TRY(cudaMemcpyAsync(ws + L.in + row_off * stride * 2, static_cast<const uint16_t*>(qkv) + r0 * stride,
                                     bytes, cudaMemcpyHostToDevice, h2d));
            if (positions)
                H3QK_TRY(cudaMemcpyAsync(ws + L.pos + row_off * o.n_axes * 4, positions + r0 * o.n_axes,
                                         c.n * o.n_axes * 4, cudaMemcpyHostToDevice, h2d));
            H3QK_TRY(cudaEventRecord(hs->in[k % kHostSlots], h2d));
            H3QK_TRY(cudaStreamWaitEvent(cmp, hs->in[k % kHostSlots], 0));
            Plan pl;
            if ((s = plan_inputs(ws + L.in + row_off * stride * 2, w_dev, w_dev + D,
                                 positions ? reinterpret_cast<const int32_t*>(ws + L.pos + row_off * o.n_axes * 4)
                                           : nullptr,
                                 c.n, heads, head_dim, rotary_dim, c.n, in_dtype, oc, cmp, &pl)) != H3QK_OK)
                return s;
            pl.p.amax_words = amax_dev;
            H3QK_TRY(launch(pl.bf16, pl.P, h3qk::kAmax, pl.p, cmp));
            row_off += c.n;
        }
        // Pass 2: cast each chunk into an output slot, copy it out.
        for (int64_t k = 0; k < n_chunks; ++k) {
            const Chunk& c = chunks[k];
            const int so = static_cast<int>(k % kHostSlots);
            if (k >= kHostSlots) H3QK_TRY(cudaStreamWaitEvent(cmp, hs->out[so], 0));
            s = h3qk_cast(ws + L.in + offs[k] * stride * 2, w_dev, w_dev + D,
                          positions ? reinterpret_cast<const int32_t*>(ws + L.pos + offs[k] * o.n_axes * 4) : nullptr,
                          c.n, heads, head_dim, rotary_dim, c.n, reinterpret_cast<const float*>(amax_dev),
                          out_ptr(so, 0), out_ptr(so, 1), out_ptr(so, 2), scales_dev, &oc, cmp);
            if (s != H3QK_OK) return s;
            H3QK_TRY(cudaEventRecord(hs->cmp[so], cmp));
            H3QK_TRY(cudaStreamWaitEvent(d2h, hs->cmp[so], 0));
            H3QK_TRY(copy_out(c.b, c.a, c.n, so));
            H3QK_TRY(cudaEventRecord(hs->out[so], d2h));
        }
    } else {
        for (int64_t k = 0; k < n_chunks; ++k) {
            const Chunk& c = chunks[k];
            const int sl = static_cast<int>(k % kHostSlots);
            if (k >= kHostSlots) H3QK_TRY(cudaStreamWaitEvent(h2d, hs->cmp[sl], 0));  // input slot free
            H3QK_TRY(copy_in(c.b, c.a, c.n, sl));
            H3QK_TRY(cudaEventRecord(hs->in[sl], h2d));
            H3QK_TRY(cudaStreamWaitEvent(cmp, hs->in[sl], 0));
            if (k >= kHostSlots) H3QK_TRY(cudaStreamWaitEvent(cmp, hs->out[sl], 0));  // output slot free
            s = h3qk_prepare(ws + L.in + sl * L.in_slot, w_dev, w_dev + D,
                             positions ? reinterpret_cast<const int32_t*>(ws + L.pos + sl * L.pos_slot) : nullptr,
                             c.n, heads, head_dim, rotary_dim, c.n, out_dtype, scale_mode, out_ptr(sl, 0),
                             out_ptr(sl, 1), out_ptr(sl, 2), e4m3 ? scales_dev : nullptr, &oc, cmp);
            if (s != H3QK_OK) return s;
            H3QK_TRY(cudaEventRecord(hs->cmp[sl], cmp));
            H3QK_TRY(cudaStreamWaitEvent(d2h, hs->cmp[sl], 0));
            H3QK_TRY(copy_out(c.b, c.a, c.n, sl));
            H3QK_TRY(cudaEventRecord(hs->out[sl], d2h));
        }
    }
    if (e4m3) {
        if (n_chunks == 0) {  // no valid row: the descales of an empty call
            s = h3qk_prepare(nullptr, w_dev, w_dev + D, nullptr, 0, heads, head_dim, rotary_dim, 0, out_dtype,
                             scale_mode, nullptr, nullptr, nullptr, scales_dev, &oc, cmp);
            if (s != H3QK_OK) return s;
        }
        H3QK_TRY(cudaEventRecord(hs->last, cmp));
        H3QK_TRY(cudaStreamWaitEvent(d2h, hs->last, 0));
        H3QK_TRY(cudaMemcpyAsync(out_scales, scales_dev, 12, cudaMemcpyDeviceToHost, d2h));
    }
    // Finish: the caller's stream waits for the last copies (which follow
    // every kernel and every copy in of this call).
    H3QK_TRY(cudaEventRecord(hs->last, cmp));
    H3QK_TRY(cudaStreamWaitEvent(d2h, hs->last, 0));
    H3QK_TRY(cudaEventRecord(hs->done, d2h));
    H3QK_TRY(cudaStreamWaitEvent(caller, hs->done, 0));
#undef H3QK_TRY
    return H3QK_OK;
}

}  // extern "C"
