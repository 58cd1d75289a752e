/*
 * h3qk.h: C-ABI of libh3qk.so, the fused QK-prep path of the MiniMax-H3
 * video VAE decoder and DiT attention on one GB300 (sm_103a).
 *
 * One call turns the packed QKV projection of a batch of token rows into
 * head-major Q, K and V.  It applies a per-head RMS normalisation to Q and K,
 * a partial multi-axis rotary embedding to Q and K, and optionally a
 * per-tensor e4m3 cast (one amax pass and one cast pass with dynamic scales,
 * or a cast with a static scale table).  Rows past a valid prefix are masked.
 *
 * Pages that define the operation:
 *  - TensorRT-LLM pull request #21485, "cuDNN FP8 attention path for
 *    MiniMax-H3 on SM107 under Ulysses": Summary, bullet 2 (the operation
 *    below, whose e4m3 form takes two kernels, a max reduction and then the
 *    conversion, with the scales computed per call or read from a table), and the
 *    commits that add the fused cast from the packed QKV projection, the
 *    single-tensor norm_rope_tensor variant (identity for V), the per-item
 *    valid length left out of the amax, and the custom-op aliasing fix
 *    (an output never aliases an input).
 *  - vllm-omni pull request #6607, MiniMax-H3 VAE decoder eager operators,
 *    "Operations" table, row "Q/K normalization + RoPE": a fixed RMS
 *    reduction order and explicit rounding points, bit-exact results.
 *  - stable-diffusion.cpp pull request #19, "MiniMax-H3: sage takes the fused
 *    RoPE op, faster video and audio VAE decode": q/k/v chunk-copied out of
 *    the fused projection, the partial RoPE, the head-major
 *    [head_dim, tokens, heads, batch] output and the fused per-head norm.
 *
 * Arithmetic (identical, bit for bit, to the CPU oracle of the test-suite):
 *   per row r < tokens with (r mod S) < valid_len, head h, t in {Q, K}:
 *     x[d]  = the 16-bit input widened to binary32;
 *     ss    = sum of x[d]^2: chunks of 8 channels summed left to right, the
 *             D/8 chunk sums (padded with zeros to a power of two) added by a
 *             halving tree p[i] += p[i + o], o = P/2 ... 1;
 *     inv   = 1 / sqrt(ss / D + eps), each operation correctly rounded;
 *     n[d]  = round16((x[d] * inv) * w_t[d]);
 *     pairs (2i, 2i+1) of the first rotary_dim channels, cut into n_axes
 *     segments of widths axis_dims[a], rotate by
 *       ang = pos[r][a] * theta^(-2i'/axis_dims[a]), i' the pair index
 *             within its segment (inverse frequency rounded to binary32
 *             once on the host),
 *       (u, v) -> (round16(u cos - v sin), round16(u sin + v cos)),
 *     with sin/cos from the library's own Cody-Waite + Taylor routine;
 *     channels >= rotary_dim pass through; V is copied unchanged.
 *   e4m3: amax_t = max |y| over the 16-bit results of the valid rows;
 *     dynamic: scale_t = amax_t / 448, factor = 448 / amax_t; static:
 *     scale_t = table[t], factor = 1 / table[t]; a zero, subnormal,
 *     infinite or NaN amax or table entry gives scale = factor = 1;
 *     code = e4m3 round-to-nearest-even, saturating at +-448, of y * factor.
 */
#ifndef H3QK_H
#define H3QK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream).  NULL is the legacy default
 * stream of the calling thread's current device. */
typedef struct CUstream_st* h3qk_stream_t;

typedef enum h3qk_status {
    H3QK_OK = 0,
    H3QK_ERR_INVALID_ARG = 1, /* a null pointer, a size or option out of range */
    H3QK_ERR_MISALIGNED = 2,  /* a pointer or row stride breaks the alignment rules */
    H3QK_ERR_ALIAS = 3,       /* an output overlaps an input or another output */
    H3QK_ERR_CUDA = 4         /* the CUDA runtime refused a launch; see h3qk_last_cuda_error */
} h3qk_status;

typedef enum h3qk_dtype {
    H3QK_DTYPE_DEFAULT = 0, /* in h3qk_opts.in_dtype only: see there */
    H3QK_FP16 = 1,          /* IEEE binary16 */
    H3QK_BF16 = 2,          /* bfloat16 */
    H3QK_E4M3 = 3           /* OCP 8-bit E4M3FN codes (output only) */
} h3qk_dtype;

typedef enum h3qk_scale_mode {
    H3QK_SCALE_NONE = 0,    /* 16-bit output, no cast */
    H3QK_SCALE_DYNAMIC = 1, /* amax pass, then cast with amax / 448 */
    H3QK_SCALE_STATIC = 2   /* cast with the caller's descale table */
} h3qk_scale_mode;

/* Optional arguments.  Pass NULL for all defaults, or fill one with
 * h3qk_opts_init() and change fields.  Enum-valued fields are int32_t. */
typedef struct h3qk_opts {
    int32_t in_dtype;        /* h3qk_dtype of qkv: H3QK_FP16 or H3QK_BF16.
                                DEFAULT: out_dtype when that is 16-bit, else BF16 */
    int32_t n_axes;          /* 3: (t, h, w) positions; 1: 1-D positions.  Default 3 */
    int32_t axis_dims[3];    /* widths of the rotary segments, even, summing to
                                rotary_dim.  All zero (default): rotary_dim/3 each
                                (n_axes 3) or rotary_dim (n_axes 1) */
    float eps;               /* RMSNorm epsilon, default 1e-6 */
    int64_t batch;           /* B >= 1: tokens = B * S rows, S rows per item.
                                valid_len applies to every item.  Default 1 */
    int64_t qkv_row_stride;  /* elements between consecutive packed rows; a
                                multiple of 8, >= 3*heads*head_dim.  0 (default):
                                3*heads*head_dim */
    double theta;            /* rotary base, default 10000 */
    const float* static_scales; /* device float[3], descales (q, k, v); required
                                   when scale_mode is STATIC, read by the kernel */
    void* workspace;         /* device memory of >= h3qk_workspace_bytes() bytes,
                                16-byte aligned, required when scale_mode is
                                DYNAMIC; holds the amax words of one call, so
                                calls that may overlap need their own.  The
                                call zeroes it on the stream, so it must not
                                overlap any input, output, the static table
                                or sat_counts (H3QK_ERR_ALIAS otherwise) */
    size_t workspace_bytes;  /* size of workspace */
    int32_t out_layout;      /* h3qk_layout of out_q/out_k/out_v: HEAD_MAJOR
                                [B, H, S, D] (default) or TOKEN_MAJOR [B, S, H, D] */
    const int32_t* valid_lens; /* device int32[batch] or NULL: item b keeps rows
                                  s < valid_lens[b] (clamped to [0, S]) instead of
                                  valid_len (which must still lie in [0, S]) */
    uint32_t* sat_counts;    /* device uint32[3] or NULL; e4m3 casts ADD to
                                sat_counts[t] the number of tensor t's values
                                whose scaled magnitude exceeds 448 (clipped to
                                the largest code).  The caller zeroes them.
                                Disjoint from every input, output and the
                                workspace (H3QK_ERR_ALIAS otherwise).
                                A counting cast runs its own kernel instance,
                                a few percent slower than the plain cast; the
                                codes and scales are the same. */
} h3qk_opts;

typedef enum h3qk_layout {
    H3QK_LAYOUT_HEAD_MAJOR = 0,  /* [B, H, S, D] */
    H3QK_LAYOUT_TOKEN_MAJOR = 1  /* [B, S, H, D] */
} h3qk_layout;

typedef enum h3qk_tensor_kind {
    H3QK_TENSOR_Q = 0, /* norm (with its weight) + RoPE */
    H3QK_TENSOR_K = 1, /* norm (with its weight) + RoPE */
    H3QK_TENSOR_V = 2  /* passed through */
} h3qk_tensor_kind;

/* Fill *opts with the defaults listed above. */
void h3qk_opts_init(h3qk_opts* opts);

/* Bytes of device workspace a DYNAMIC call needs (16). */
size_t h3qk_workspace_bytes(void);

/*
 * h3qk_prepare: the whole path for one batch of packed QKV rows.
 *
 * Arguments (every pointer is device memory owned by the caller; the library
 * allocates nothing and keeps no pointer after the call returns):
 *   qkv        16-bit [tokens, row_stride] row-major, row r = [Q | K | V],
 *              each heads*head_dim values with head h's channels at
 *              h*head_dim; 16-byte aligned.  Read only.
 *   norm_wq    float[head_dim], RMSNorm weight of Q, shared by the heads;
 *              16-byte aligned.  Read only.
 *   norm_wk    float[head_dim], RMSNorm weight of K; 16-byte aligned.
 *   positions  int32 [tokens, n_axes] row-major: each row's position on each
 *              axis (tile-local grid indices, or 0..S-1 for 1-D).  May be
 *              NULL when rotary_dim is 0.  Read only.
 *   tokens     B*S >= 0 rows.  0 is a valid empty call: qkv, positions and
 *              the three row outputs may then be NULL; in e4m3 modes the
 *              descales are still written (1 for DYNAMIC, the table for
 *              STATIC).
 *   heads      H >= 1.
 *   head_dim   D: a multiple of 8 in [8, 256].
 *   rotary_dim R: even, 0 <= R <= D.
 *   valid_len  0 <= valid_len <= S: rows s >= valid_len of every item are
 *              neither read for the amax nor written.
 *   out_dtype  H3QK_FP16 / H3QK_BF16 (must equal the input type) with
 *              scale_mode NONE, or H3QK_E4M3 with DYNAMIC or STATIC.
 *   out_q, out_k, out_v  [B, H, S, D] (or [B, S, H, D], opts->out_layout)
 *              contiguous, 2 bytes (16-bit) or 1 byte (e4m3) per element;
 *              16-byte aligned; pairwise disjoint and disjoint from every
 *              input, from the static table, the workspace and the
 *              counters.  Rows past valid_len keep their previous bytes.
 *   out_scales float[3] descales (q, k, v) written in e4m3 modes (NULL
 *              allowed with scale_mode NONE); never the static table itself.
 *   opts       NULL or see h3qk_opts.
 *   stream     the stream the kernels are enqueued on.
 *
 * Errors: every argument is checked on the host before anything is
 * enqueued; a check that fails returns its status and enqueues nothing.
 * H3QK_ERR_CUDA reports a failed launch (h3qk_last_cuda_error() gives the
 * CUDA error code of the calling thread's last failure).  The call is
 * asynchronous on `stream`: it never synchronises, never aborts and never
 * traps; results are ready when the stream reaches them.
 */
h3qk_status h3qk_prepare(const void* qkv, const float* norm_wq, const float* norm_wk,
                         const int32_t* positions, int64_t tokens, int32_t heads,
                         int32_t head_dim, int32_t rotary_dim, int64_t valid_len,
                         h3qk_dtype out_dtype, h3qk_scale_mode scale_mode, void* out_q,
                         void* out_k, void* out_v, float* out_scales, const h3qk_opts* opts,
                         h3qk_stream_t stream);

/*
 * h3qk_norm_rope_tensor: the same path for one separately projected tensor
 * [B, S, H, D] (rows of H*D values, row stride opts->qkv_row_stride or H*D):
 * per-head RMS norm with norm_w and the partial RoPE for kind Q or K, the
 * identity for kind V (norm_w may then be NULL); 16-bit output (the input
 * type) or e4m3 with the tensor's own descale (out_scale, float[1]; dynamic
 * from its amax over the valid rows, using opts->workspace; static from
 * opts->static_scales[0]).  The output keeps the input's token-major
 * [B, S, H, D] layout (opts->out_layout is ignored).  This is the
 * single-tensor form of the pages' fused cast for the path that projects Q,
 * K and V separately (TensorRT-LLM PR #21485, commit adding
 * norm_rope_tensor(x, norm_weight, cos, sin, eps, fp8=...)).  Errors and
 * asynchrony as for h3qk_prepare.
 */
h3qk_status h3qk_norm_rope_tensor(const void* x, const float* norm_w, const int32_t* positions,
                                  int64_t tokens, int32_t heads, int32_t head_dim,
                                  int32_t rotary_dim, int64_t valid_len, h3qk_tensor_kind kind,
                                  h3qk_dtype out_dtype, h3qk_scale_mode scale_mode, void* out,
                                  float* out_scale, const h3qk_opts* opts, h3qk_stream_t stream);

/*
 * h3qk_amax and h3qk_cast: the two passes of a DYNAMIC e4m3 call, separately,
 * so that a caller whose rows are sharded over several GPUs can all-reduce
 * (MAX) the three amax values between them and cast every shard with the
 * same scales.  This is the exchange the pages make under Ulysses sequence
 * parallelism (TensorRT-LLM PR #21485, the commit that all-reduces the amax
 * so that all ranks share one scale per tensor).  On one GPU,
 * h3qk_amax followed by h3qk_cast on the same stream gives the same bytes as
 * h3qk_prepare with H3QK_SCALE_DYNAMIC.
 *
 * The input arguments are those of h3qk_prepare; opts->in_dtype DEFAULT means
 * BF16 here, and opts->static_scales / workspace are ignored.
 *
 * h3qk_amax writes out_amax (device float[3], 4-byte aligned): the largest
 * |y| of Q, K and V over the valid rows, y the 16-bit value h3qk_prepare
 * would write (0 when no row is valid).  It zeroes out_amax first, on the
 * stream, then accumulates into it with atomics.
 *
 * h3qk_cast reads amax (device float[3]; after any all-reduce), derives the
 * dynamic scales from it as h3qk_prepare does (scale = amax / 448, factor =
 * 448 / amax; 1 and 1 for a zero, subnormal, infinite or NaN amax) and writes
 * the e4m3 codes of the valid rows into out_q, out_k, out_v and the three
 * descales into out_scales.  Outputs must not overlap the inputs, amax or
 * each other.
 *
 * Errors and asynchrony as for h3qk_prepare.
 */
h3qk_status h3qk_amax(const void* qkv, const float* norm_wq, const float* norm_wk,
                      const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                      int32_t rotary_dim, int64_t valid_len, float* out_amax, const h3qk_opts* opts,
                      h3qk_stream_t stream);

h3qk_status h3qk_cast(const void* qkv, const float* norm_wq, const float* norm_wk,
                      const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                      int32_t rotary_dim, int64_t valid_len, const float* amax, void* out_q,
                      void* out_k, void* out_v, float* out_scales, const h3qk_opts* opts,
                      h3qk_stream_t stream);

/*
 * h3qk_prepare_sage: the path with the outputs a sage attention kernel reads
 * (stable-diffusion.cpp PR #19, first commit: the fused RoPE / permute op
 * writes head-major [head_dim, tokens, heads, batch] tensors, F32 Q, F32 K
 * times kv_scale and F16 V times kv_scale, with the rounding points of the
 * unfused sage chain).
 *
 * Arithmetic: the widened 16-bit input stays binary32 to the end: the
 * normalised value (x * inv) * w is NOT rounded to 16 bits before the
 * rotation; the rotated values are written as binary32 for Q, and as
 * binary32 products with kv_scale (one rounding) for K; V is widened,
 * multiplied by kv_scale (one binary32 rounding) and rounded to binary16
 * (nearest even, overflow to infinity).  Norm, reduction tree, sin/cos and
 * angles are those of h3qk_prepare.
 *
 * Arguments as for h3qk_prepare, except:
 *   kv_scale   a finite binary32 factor of K and V (1 leaves them unscaled).
 *   out_q, out_k  float [B, H, S, D] (or [B, S, H, D], opts->out_layout).
 *   out_v      IEEE binary16 codes, same shape.
 *   All three 16-byte aligned, pairwise disjoint and disjoint from every
 *   input; rows past the valid prefix keep their previous bytes.
 *   opts->in_dtype DEFAULT means BF16; opts->static_scales, workspace and
 *   sat_counts are ignored (there is no e4m3 cast).
 * Errors and asynchrony as for h3qk_prepare (a non-finite kv_scale is
 * H3QK_ERR_INVALID_ARG).
 */
h3qk_status h3qk_prepare_sage(const void* qkv, const float* norm_wq, const float* norm_wk,
                              const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                              int32_t rotary_dim, int64_t valid_len, float kv_scale, float* out_q,
                              float* out_k, void* out_v, const h3qk_opts* opts, h3qk_stream_t stream);

/*
 * h3qk_prepare_host: h3qk_prepare on HOST buffers.  The inputs (qkv,
 * norm_wq, norm_wk, positions, opts->static_scales, opts->valid_lens) and
 * the outputs (out_q, out_k, out_v, out_scales) are host memory, laid out as
 * for h3qk_prepare; page-locked (pinned) memory lets the copies run
 * asynchronously and overlap, pageable memory works but serialises them.
 * The pages move the fused op's inputs and outputs as device tensors; this
 * entry adds the transfers for callers whose tensors live on the host, the
 * whole round trip being one library call.
 *
 * The call is cut into chunks of about 64 MiB of input rows (256 to 8,192
 * token rows) inside one item.
 * Three streams owned by the library (created on the first call on each
 * device) copy a chunk in, compute it and copy it out, so the transfers of
 * one chunk overlap the kernels and transfers of others.  In dynamic e4m3
 * mode every chunk goes through the amax pass as it arrives and the cast
 * pass follows once all have arrived.  Only valid rows are copied: output
 * rows past the valid prefix keep their previous bytes on the host.
 *
 *   workspace        device memory, 256-byte aligned, of at least
 *                    h3qk_host_workspace_bytes() bytes for this call shape:
 *                    the weights, a ring of three chunk slots (dynamic
 *                    e4m3: the whole input, which the cast pass reads after
 *                    the amax pass) and the descales.  Calls that share a
 *                    workspace must be ordered (one caller stream).
 *   opts             as for h3qk_prepare, except that static_scales and
 *                    valid_lens are host arrays, and sat_counts and
 *                    opts->workspace must be NULL.
 *   stream           the call starts after the work already enqueued on it,
 *                    and work enqueued on it afterwards starts after the
 *                    call's last copy; the host buffers must stay valid and
 *                    unchanged until then.  The call returns after enqueuing
 *                    (synchronise the stream before reading the outputs).
 * Errors as for h3qk_prepare; a workspace that is too small is
 * H3QK_ERR_INVALID_ARG.  Host calls on one device enqueue one at a time.
 */
size_t h3qk_host_workspace_bytes(int64_t tokens, int32_t heads, int32_t head_dim, h3qk_dtype out_dtype,
                                 h3qk_scale_mode scale_mode, const h3qk_opts* opts);

h3qk_status h3qk_prepare_host(const void* qkv, const float* norm_wq, const float* norm_wk,
                              const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                              int32_t rotary_dim, int64_t valid_len, h3qk_dtype out_dtype,
                              h3qk_scale_mode scale_mode, void* out_q, void* out_k, void* out_v,
                              float* out_scales, const h3qk_opts* opts, void* workspace,
                              size_t workspace_bytes, h3qk_stream_t stream);

/*
 * h3qk_prepare_noalloc: h3qk_prepare for callers that cannot allocate device
 * memory at the point of the call -- for example a plugin inside an inference
 * engine that receives all of its memory up front, or a real-time decode loop
 * whose memory budget is fixed at start-up.  The pages have no counterpart to
 * this entry point; it is a property of this library only.
 *
 * Arguments, results and errors are those of h3qk_prepare, except that a
 * DYNAMIC call ignores opts->workspace and keeps its amax words in a fixed
 * scratch array inside the library (a file-scope __device__ array of 256
 * bytes, 256-byte aligned, held by every GPU that loads the library until the
 * process exits).  A call needs 16 bytes of it whatever its sizes; a call
 * that needed more than the array holds would be rejected with
 * H3QK_ERR_INVALID_ARG.  The call allocates nothing and calls no allocating
 * routine.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 * capture on that device.  Every call shares the one array, which keeps the
 * last call's contents (each DYNAMIC call clears its amax words first), so
 * DYNAMIC calls whose kernels overlap on the GPU (different streams, no
 * ordering between them) race on it: order them on one stream, or use
 * h3qk_prepare with a workspace per stream.
 */
h3qk_status h3qk_prepare_noalloc(const void* qkv, const float* norm_wq, const float* norm_wk,
                                 const int32_t* positions, int64_t tokens, int32_t heads,
                                 int32_t head_dim, int32_t rotary_dim, int64_t valid_len,
                                 h3qk_dtype out_dtype, h3qk_scale_mode scale_mode, void* out_q,
                                 void* out_k, void* out_v, float* out_scales,
                                 const h3qk_opts* opts, h3qk_stream_t stream);

/*
 * Adjacent operations of the MiniMax-H3 VAE decoder block (vllm-omni PR #6607,
 * "Operations" table, rows "SwiGLU" and "Scaled residual"): streaming,
 * HBM-bound, bit-exact to the test-suite's CPU oracle.
 *
 * h3qk_silu_and_mul: x is [rows, row_stride] 16-bit (dtype FP16 or BF16)
 * holding gate = x[:, 0:f] and up = x[:, f:2f] (row_stride 0 means 2f; a
 * multiple of 8); out is [rows, f] of the same type:
 *   out = round16(silu(gate) * up),  silu(g) = g / (1 + e^-g),
 * with a rounded sum, a correctly rounded division, a rounded product, and
 * the library's own e^x (Cody-Waite reduction + Taylor series; the same
 * routine as the oracle).  f is a multiple of 8; x and out 16-byte aligned
 * and disjoint.
 *
 * h3qk_scaled_residual: out[r, c] = residual[r, c] + branch[r, c] * scale[c]
 * (scale_len == channels) or * scale[0] (scale_len == 1); residual, out and
 * scale are FP32, branch 16-bit (branch_dtype); the product is rounded on its
 * own, then the sum (no multiply-add contraction).  channels is a multiple of 8;
 * residual, branch, out (and a vector scale) 16-byte aligned; out may be
 * residual itself (in place) but must not otherwise overlap an input.
 *
 * Errors and asynchrony as for h3qk_prepare.
 */
h3qk_status h3qk_silu_and_mul(const void* x, h3qk_dtype dtype, int64_t rows, int32_t f, int64_t row_stride,
                              void* out, h3qk_stream_t stream);

h3qk_status h3qk_scaled_residual(const float* residual, const void* branch, h3qk_dtype branch_dtype,
                                 const float* scale, int64_t rows, int32_t channels, int32_t scale_len,
                                 float* out, h3qk_stream_t stream);

/* A static, human-readable name of a status. */
const char* h3qk_status_string(h3qk_status status);

/* The cudaError_t code of the calling thread's last H3QK_ERR_CUDA (0 if none). */
int h3qk_last_cuda_error(void);

/* Number of kernel launches the calling thread's h3qk calls have enqueued
 * since the last reset (evidence that the CUDA path ran); reset with
 * h3qk_launch_count_reset(). */
uint64_t h3qk_launch_count(void);
void h3qk_launch_count_reset(void);

/* Library version, major*10000 + minor*100 + patch. */
int h3qk_version(void);

/*
 * Debug builds.  `python -m video_vae_decoder_qkv_gb300.build --debug` builds
 * libh3qk_debug.so with device-side bounds checks, in place of a memory
 * sanitizer.  Every
 * global load, store and atomic of the QK-prep kernels is checked against
 * the extent of its buffer first.  A failed check is recorded in status
 * words on the device and the access is skipped; nothing traps.
 *
 * h3qk_debug_checks: 1 in a debug build, 0 in the release library.
 * h3qk_debug_status: copies the current device's four status words to
 *   out[4] (synchronous; waits for all work on the device to finish):
 *   out[0] the OR of the failed checks (1 packed-row load, 2 output store,
 *   4 position load, 8 per-item length load, 16 amax word / descale /
 *   counter index), out[1] the number of failures, out[2..3] the first
 *   failing element offset + 1 as a little-endian 64-bit value (0: none).
 *   With reset != 0 it then zeroes them.  H3QK_ERR_INVALID_ARG in a release
 *   build or for a NULL out.
 * h3qk_debug_limit_outputs: a test hook.  elements >= 0 makes later calls
 *   of this process treat each output tensor as holding at most `elements`
 *   elements, so the checks report and skip the stores past it; a negative
 *   value restores the calls' own extents.  No effect in a release build.
 */
int h3qk_debug_checks(void);
h3qk_status h3qk_debug_status(uint32_t* out, int reset);
void h3qk_debug_limit_outputs(int64_t elements);

#ifdef __cplusplus
}
#endif

#endif /* H3QK_H */
