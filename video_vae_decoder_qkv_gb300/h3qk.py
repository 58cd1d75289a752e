"""Python binding of libh3qk.so (ctypes).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  When the
library has not been built this module raises instead of computing anything
another way.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libh3qk.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "h3qk.h")

DTYPE_DEFAULT, FP16, BF16, E4M3 = 0, 1, 2, 3
SCALE_NONE, SCALE_DYNAMIC, SCALE_STATIC = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_MISALIGNED, ERR_ALIAS, ERR_CUDA = 0, 1, 2, 3, 4
HEAD_MAJOR, TOKEN_MAJOR = 0, 1
TENSOR_Q, TENSOR_K, TENSOR_V = 0, 1, 2
_SCALE_NAMES = {"none": SCALE_NONE, "dynamic": SCALE_DYNAMIC, "static": SCALE_STATIC}


class H3QKError(RuntimeError):
    def __init__(self, status: int, name: str, cuda_error: int = 0):
        msg = f"h3qk_prepare failed: {name} (status {status})"
        if status == ERR_CUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)
        self.status = status
        self.cuda_error = cuda_error


class Opts(ctypes.Structure):
    """Mirror of h3qk_opts (include/h3qk.h)."""

    _fields_ = [
        ("in_dtype", ctypes.c_int32),
        ("n_axes", ctypes.c_int32),
        ("axis_dims", ctypes.c_int32 * 3),
        ("eps", ctypes.c_float),
        ("batch", ctypes.c_int64),
        ("qkv_row_stride", ctypes.c_int64),
        ("theta", ctypes.c_double),
        ("static_scales", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("out_layout", ctypes.c_int32),
        ("valid_lens", ctypes.c_void_p),
        ("sat_counts", ctypes.c_void_p),
    ]


_lib = None


def load_library(path: str) -> ctypes.CDLL:
    """Load a build of the library at `path` with the C signatures set (the
    release libh3qk.so through lib(), or the debug build libh3qk_debug.so)."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m video_vae_decoder_qkv_gb300.build` "
            "(or __graft_entry__.build()); there is no other implementation of this path")
    L = ctypes.CDLL(path)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.h3qk_prepare.restype = ctypes.c_int
    L.h3qk_prepare.argtypes = [P, P, P, P, I64, I32, I32, I32, I64, ctypes.c_int, ctypes.c_int,
                               P, P, P, P, ctypes.POINTER(Opts), P]
    L.h3qk_opts_init.restype = None
    L.h3qk_opts_init.argtypes = [ctypes.POINTER(Opts)]
    L.h3qk_workspace_bytes.restype = ctypes.c_size_t
    L.h3qk_status_string.restype = ctypes.c_char_p
    L.h3qk_status_string.argtypes = [ctypes.c_int]
    L.h3qk_last_cuda_error.restype = ctypes.c_int
    L.h3qk_launch_count.restype = ctypes.c_uint64
    L.h3qk_launch_count_reset.restype = None
    L.h3qk_version.restype = ctypes.c_int
    L.h3qk_debug_checks.restype = ctypes.c_int
    L.h3qk_debug_status.restype = ctypes.c_int
    L.h3qk_debug_status.argtypes = [P, ctypes.c_int]
    L.h3qk_debug_limit_outputs.restype = None
    L.h3qk_debug_limit_outputs.argtypes = [I64]
    return L


def lib() -> ctypes.CDLL:
    """Load libh3qk.so; raise if it was not built."""
    global _lib
    if _lib is None:
        _lib = load_library(LIB_PATH)
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/h3qk.h declares."""
    with open(HEADER) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(h3qk_[a-z0-9_]+)\s*\(", src)))


def default_opts() -> Opts:
    o = Opts()
    lib().h3qk_opts_init(ctypes.byref(o))
    return o


def status_string(status: int) -> str:
    return lib().h3qk_status_string(status).decode()


def launch_count() -> int:
    return int(lib().h3qk_launch_count())


def launch_count_reset() -> None:
    lib().h3qk_launch_count_reset()


def prepare_ptr(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim, valid_len,
                out_dtype, scale_mode, out_q, out_k, out_v, out_scales, opts: Opts | None, stream) -> int:
    """Call h3qk_prepare with raw integer addresses; returns the status."""
    L = lib()
    return int(L.h3qk_prepare(qkv, norm_wq, norm_wk, positions, int(tokens), int(heads),
                              int(head_dim), int(rotary_dim), int(valid_len), int(out_dtype),
                              int(scale_mode), out_q, out_k, out_v, out_scales,
                              ctypes.byref(opts) if opts is not None else None, stream))


def prepare_noalloc_ptr(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                        valid_len, out_dtype, scale_mode, out_q, out_k, out_v, out_scales,
                        opts: Opts | None, stream) -> int:
    """Call h3qk_prepare_noalloc (for callers that cannot allocate device
    memory: a DYNAMIC call keeps its amax words in the library's own fixed
    scratch array) with raw integer addresses; returns the status."""
    L = lib()
    fn = L.h3qk_prepare_noalloc
    if fn.argtypes is None:
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        fn.restype = ctypes.c_int
        fn.argtypes = [P, P, P, P, I64, I32, I32, I32, I64, ctypes.c_int, ctypes.c_int,
                       P, P, P, P, ctypes.POINTER(Opts), P]
    return int(fn(qkv, norm_wq, norm_wk, positions, int(tokens), int(heads), int(head_dim),
                  int(rotary_dim), int(valid_len), int(out_dtype), int(scale_mode), out_q, out_k,
                  out_v, out_scales, ctypes.byref(opts) if opts is not None else None, stream))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, *, device=None, esz=None, dtypes=None, numel=None, min_numel=None, optional=False):
    """Reject a caller tensor that does not fit what the library will read or
    write through its pointer: the C-ABI sees only addresses, so a short or
    strided buffer would be overrun on the device."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if esz is not None and t.element_size() != esz:
        raise TypeError(f"{name} must have {esz}-byte elements, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name} must have at least {min_numel} elements, got {t.numel()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _need_rows(x, name, width):
    """A packed input [tokens, row_stride] whose rows hold `width` values."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D [tokens, row_stride] with unit inner stride")
    if x.shape[1] < width:
        raise ValueError(f"{name} rows hold {x.shape[1]} values, the call reads {width}")


def _need_common(qkv, norm_wq, norm_wk, positions, *, tokens, heads, head_dim, rotary_dim, n_axes, batch,
                 valid_lens, device, width_parts=3, weights=("norm_wq", "norm_wk")):
    import torch

    _need_rows(qkv, "qkv", width_parts * heads * head_dim)
    for w, name in zip((norm_wq, norm_wk), weights):
        _need(w, name, device=device, dtypes=(torch.float32,), numel=head_dim)
    if positions is not None or rotary_dim > 0:
        _need(positions, "positions", device=device, dtypes=(torch.int32,), numel=tokens * n_axes)
    _need(valid_lens, "valid_lens", device=device, dtypes=(torch.int32,), numel=batch, optional=True)


def prepare(qkv, norm_wq, norm_wk, positions, *, heads: int, head_dim: int, rotary_dim: int,
            batch: int = 1, valid_len: int | None = None, scale_mode: str = "none",
            n_axes: int | None = None, axis_dims=None, theta: float = 10000.0, eps: float = 1e-6,
            static_scales=None, out=None, out_scales=None, workspace=None, stream=None,
            out_layout: str = "head_major", valid_lens=None, sat_counts=None):
    """The fused QK-prep path on torch CUDA tensors.

    qkv: fp16/bf16 [tokens, row_stride] (row stride a multiple of 8 elements,
    >= 3*heads*head_dim); norm_wq / norm_wk: float32 [head_dim]; positions:
    int32 [tokens, n_axes].  scale_mode: "none" (16-bit out, the input type),
    "dynamic" or "static" (e4m3 out; static needs ``static_scales``, a
    float32 [3] CUDA tensor of descales).  Returns (q, k, v, scales): q, k, v
    head-major [batch, heads, S, head_dim], scales a float32 [3] tensor of
    descales in e4m3 modes, else None.  ``out``, ``out_scales`` and
    ``workspace`` reuse caller buffers (rows past valid_len of ``out`` keep
    their contents).  ``out_layout="token_major"`` writes [batch, S, heads,
    head_dim]; ``valid_lens`` (int32 [batch] CUDA tensor) gives each item its
    own valid length; ``sat_counts`` (int32/uint32 [3] CUDA tensor, zeroed by
    the caller) receives the e4m3 saturation counts.
    """
    import torch

    if qkv.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("qkv must be float16 or bfloat16")
    if qkv.dim() != 2 or qkv.stride(1) != 1:
        raise ValueError("qkv must be 2-D [tokens, row_stride] with unit inner stride")
    tokens = qkv.shape[0]
    if tokens % batch:
        raise ValueError("tokens must be a multiple of batch")
    seq = tokens // batch
    if valid_len is None:
        valid_len = seq
    mode = _SCALE_NAMES[scale_mode]
    in_dt = FP16 if qkv.dtype == torch.float16 else BF16
    out_dt = in_dt if mode == SCALE_NONE else E4M3
    if n_axes is None:
        n_axes = positions.shape[1] if positions is not None and positions.dim() == 2 else 3
    dev = qkv.device
    layout = {"head_major": HEAD_MAJOR, "token_major": TOKEN_MAJOR}[out_layout]
    shape = (batch, heads, seq, head_dim) if layout == HEAD_MAJOR else (batch, seq, heads, head_dim)
    _need_common(qkv, norm_wq, norm_wk, positions, tokens=tokens, heads=heads, head_dim=head_dim,
                 rotary_dim=rotary_dim, n_axes=n_axes, batch=batch, valid_lens=valid_lens, device=dev)
    if out is None:
        tdt = qkv.dtype if out_dt != E4M3 else torch.float8_e4m3fn
        out = tuple(torch.empty(shape, dtype=tdt, device=dev) for _ in range(3))
    q, k, v = out
    for t, name in zip((q, k, v), ("out[0]", "out[1]", "out[2]")):
        _need(t, name, device=dev, esz=1 if out_dt == E4M3 else 2, numel=tokens * heads * head_dim)
    if out_dt == E4M3 and out_scales is None:
        out_scales = torch.empty(3, dtype=torch.float32, device=dev)
    if out_dt == E4M3:
        _need(out_scales, "out_scales", device=dev, dtypes=(torch.float32,), min_numel=3)
    if mode == SCALE_STATIC:
        _need(static_scales, "static_scales", device=dev, dtypes=(torch.float32,), min_numel=3)
    _need(sat_counts, "sat_counts", device=dev, esz=4, min_numel=3, optional=True)
    _need(workspace, "workspace", device=dev, optional=True)
    if mode == SCALE_DYNAMIC and workspace is None:
        workspace = torch.empty(int(lib().h3qk_workspace_bytes()) // 4, dtype=torch.int32, device=dev)
    o = default_opts()
    o.in_dtype = in_dt
    o.n_axes = n_axes
    if axis_dims is not None:
        dims = list(axis_dims) + [0] * (3 - len(axis_dims))
        o.axis_dims = (ctypes.c_int32 * 3)(*dims)
    o.eps = eps
    o.batch = batch
    o.qkv_row_stride = qkv.stride(0)
    o.theta = theta
    o.static_scales = _ptr(static_scales)
    o.out_layout = layout
    o.valid_lens = _ptr(valid_lens)
    o.sat_counts = _ptr(sat_counts)
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(dev):  # the library keys its caches on the current device
        st = prepare_ptr(qkv.data_ptr(), norm_wq.data_ptr(), norm_wk.data_ptr(), _ptr(positions), tokens,
                         heads, head_dim, rotary_dim, valid_len, out_dt, mode, q.data_ptr(),
                         k.data_ptr(), v.data_ptr(), _ptr(out_scales) if out_dt == E4M3 else None, o, stream)
    if st != OK:
        raise H3QKError(st, status_string(st), int(lib().h3qk_last_cuda_error()))
    return q, k, v, (out_scales if out_dt == E4M3 else None)


def _sage_sig(L):
    fn = L.h3qk_prepare_sage
    if fn.argtypes is None:
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        fn.restype = ctypes.c_int
        fn.argtypes = [P, P, P, P, I64, I32, I32, I32, I64, ctypes.c_float, P, P, P,
                       ctypes.POINTER(Opts), P]
    return fn


def prepare_sage_ptr(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim, valid_len,
                     kv_scale, out_q, out_k, out_v, opts, stream) -> int:
    """h3qk_prepare_sage on raw device pointers (ints); returns the status."""
    return _sage_sig(lib())(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim,
                            valid_len, kv_scale, out_q, out_k, out_v,
                            ctypes.byref(opts) if opts is not None else None, stream)


def prepare_sage(qkv, norm_wq, norm_wk, positions, *, heads: int, head_dim: int, rotary_dim: int,
                 kv_scale: float = 1.0, batch: int = 1, valid_len: int | None = None,
                 n_axes: int | None = None, axis_dims=None, theta: float = 10000.0, eps: float = 1e-6,
                 out=None, stream=None, out_layout: str = "head_major", valid_lens=None):
    """The path with the outputs a sage attention kernel reads: float32 Q,
    float32 K * kv_scale and float16 V * kv_scale, head-major [batch, heads,
    S, head_dim] (or token-major).  Inputs as for ``prepare``.  Returns
    (q, k, v)."""
    import torch

    if qkv.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("qkv must be float16 or bfloat16")
    if qkv.dim() != 2 or qkv.stride(1) != 1:
        raise ValueError("qkv must be 2-D [tokens, row_stride] with unit inner stride")
    tokens = qkv.shape[0]
    if tokens % batch:
        raise ValueError("tokens must be a multiple of batch")
    seq = tokens // batch
    if valid_len is None:
        valid_len = seq
    if n_axes is None:
        n_axes = positions.shape[1] if positions is not None and positions.dim() == 2 else 3
    layout = {"head_major": HEAD_MAJOR, "token_major": TOKEN_MAJOR}[out_layout]
    shape = (batch, heads, seq, head_dim) if layout == HEAD_MAJOR else (batch, seq, heads, head_dim)
    dev = qkv.device
    _need_common(qkv, norm_wq, norm_wk, positions, tokens=tokens, heads=heads, head_dim=head_dim,
                 rotary_dim=rotary_dim, n_axes=n_axes, batch=batch, valid_lens=valid_lens, device=dev)
    if out is None:
        out = (torch.empty(shape, dtype=torch.float32, device=dev),
               torch.empty(shape, dtype=torch.float32, device=dev),
               torch.empty(shape, dtype=torch.float16, device=dev))
    q, k, v = out
    for t, name, esz in ((q, "out[0]", 4), (k, "out[1]", 4), (v, "out[2]", 2)):
        _need(t, name, device=dev, esz=esz, numel=tokens * heads * head_dim)
    o = _opts_for(qkv, n_axes=n_axes, axis_dims=axis_dims, theta=theta, eps=eps, batch=batch)
    o.out_layout = layout
    o.valid_lens = _ptr(valid_lens)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(dev):  # the library keys its caches on the current device
        st = prepare_sage_ptr(qkv.data_ptr(), norm_wq.data_ptr(), norm_wk.data_ptr(), _ptr(positions), tokens,
                              heads, head_dim, rotary_dim, valid_len, float(kv_scale), q.data_ptr(), k.data_ptr(),
                              v.data_ptr(), o, stream)
    if st != OK:
        raise H3QKError(st, status_string(st), int(lib().h3qk_last_cuda_error()))
    return q, k, v


def _host_sigs(L):
    if L.h3qk_prepare_host.argtypes is None:
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.h3qk_host_workspace_bytes.restype = ctypes.c_size_t
        L.h3qk_host_workspace_bytes.argtypes = [I64, I32, I32, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts)]
        L.h3qk_prepare_host.restype = ctypes.c_int
        L.h3qk_prepare_host.argtypes = [P, P, P, P, I64, I32, I32, I32, I64, ctypes.c_int, ctypes.c_int, P, P, P, P,
                                        ctypes.POINTER(Opts), P, ctypes.c_size_t, P]


def host_workspace_bytes(tokens: int, heads: int, head_dim: int, out_dtype: int, scale_mode: int, opts=None) -> int:
    L = lib()
    _host_sigs(L)
    return int(L.h3qk_host_workspace_bytes(tokens, heads, head_dim, out_dtype, scale_mode,
                                           ctypes.byref(opts) if opts is not None else None))


def prepare_host_ptr(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim, valid_len, out_dtype,
                     scale_mode, out_q, out_k, out_v, out_scales, opts, workspace, workspace_bytes, stream) -> int:
    """h3qk_prepare_host on raw pointers (host buffers, device workspace); returns the status."""
    L = lib()
    _host_sigs(L)
    return L.h3qk_prepare_host(qkv, norm_wq, norm_wk, positions, tokens, heads, head_dim, rotary_dim, valid_len,
                               out_dtype, scale_mode, out_q, out_k, out_v, out_scales,
                               ctypes.byref(opts) if opts is not None else None, workspace, workspace_bytes, stream)


def prepare_host(qkv, norm_wq, norm_wk, positions, *, heads: int, head_dim: int, rotary_dim: int,
                 batch: int = 1, valid_len: int | None = None, scale_mode: str = "none",
                 n_axes: int | None = None, axis_dims=None, theta: float = 10000.0, eps: float = 1e-6,
                 static_scales=None, out=None, out_scales=None, workspace=None, stream=None,
                 out_layout: str = "head_major", valid_lens=None, device=None):
    """The path on host (CPU) tensors, one library call: inputs are copied to
    the GPU, computed and copied back in overlapping chunks.  Arguments as for
    ``prepare``, but every tensor is a CPU tensor (pinned memory lets the
    copies overlap); ``static_scales`` and ``valid_lens`` are CPU tensors too.
    ``workspace`` is a CUDA uint8 tensor of ``host_workspace_bytes`` bytes
    (allocated when None).  Returns (q, k, v, scales) as CPU tensors; they are
    ready once ``stream`` (default: the current stream) has been
    synchronised."""
    import torch

    if qkv.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("qkv must be float16 or bfloat16")
    if qkv.device.type != "cpu":
        raise ValueError("prepare_host takes host tensors")
    tokens = qkv.shape[0]
    if tokens % batch:
        raise ValueError("tokens must be a multiple of batch")
    seq = tokens // batch
    if valid_len is None:
        valid_len = seq
    mode = _SCALE_NAMES[scale_mode]
    in_dt = FP16 if qkv.dtype == torch.float16 else BF16
    out_dt = in_dt if mode == SCALE_NONE else E4M3
    if n_axes is None:
        n_axes = positions.shape[1] if positions is not None and positions.dim() == 2 else 3
    layout = {"head_major": HEAD_MAJOR, "token_major": TOKEN_MAJOR}[out_layout]
    shape = (batch, heads, seq, head_dim) if layout == HEAD_MAJOR else (batch, seq, heads, head_dim)
    host = qkv.device
    _need_common(qkv, norm_wq, norm_wk, positions, tokens=tokens, heads=heads, head_dim=head_dim,
                 rotary_dim=rotary_dim, n_axes=n_axes, batch=batch, valid_lens=valid_lens, device=host)
    if out is None:
        tdt = qkv.dtype if out_dt != E4M3 else torch.uint8
        out = tuple(torch.empty(shape, dtype=tdt).pin_memory() for _ in range(3))
    q, k, v = out
    for t, name in zip((q, k, v), ("out[0]", "out[1]", "out[2]")):
        _need(t, name, device=host, esz=1 if out_dt == E4M3 else 2, numel=tokens * heads * head_dim)
    if out_dt == E4M3 and out_scales is None:
        out_scales = torch.empty(3, dtype=torch.float32).pin_memory()
    if out_dt == E4M3:
        _need(out_scales, "out_scales", device=host, dtypes=(torch.float32,), min_numel=3)
    if mode == SCALE_STATIC:
        _need(static_scales, "static_scales", device=host, dtypes=(torch.float32,), min_numel=3)
    o = _opts_for(qkv, n_axes=n_axes, axis_dims=axis_dims, theta=theta, eps=eps, batch=batch)
    o.out_layout = layout
    o.static_scales = _ptr(static_scales)
    o.valid_lens = _ptr(valid_lens)
    need = host_workspace_bytes(tokens, heads, head_dim, out_dt, mode, o)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(dev):  # the library keys its caches on the current device
        st = prepare_host_ptr(qkv.data_ptr(), norm_wq.data_ptr(), norm_wk.data_ptr(), _ptr(positions), tokens, heads,
                              head_dim, rotary_dim, valid_len, out_dt, mode, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                              _ptr(out_scales) if out_dt == E4M3 else None, o, workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), stream)
    if st != OK:
        raise H3QKError(st, status_string(st), int(lib().h3qk_last_cuda_error()))
    return q, k, v, (out_scales if out_dt == E4M3 else None)


def _opts_for(qkv, *, n_axes, axis_dims, theta, eps, batch):
    import torch

    o = default_opts()
    o.in_dtype = FP16 if qkv.dtype == torch.float16 else BF16
    o.n_axes = n_axes
    if axis_dims is not None:
        dims = list(axis_dims) + [0] * (3 - len(axis_dims))
        o.axis_dims = (ctypes.c_int32 * 3)(*dims)
    o.eps = eps
    o.batch = batch
    o.qkv_row_stride = qkv.stride(0)
    o.theta = theta
    return o


def _split_sigs(L):
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    if L.h3qk_amax.argtypes is None:
        L.h3qk_amax.restype = ctypes.c_int
        L.h3qk_amax.argtypes = [P, P, P, P, I64, I32, I32, I32, I64, P, ctypes.POINTER(Opts), P]
        L.h3qk_cast.restype = ctypes.c_int
        L.h3qk_cast.argtypes = [P, P, P, P, I64, I32, I32, I32, I64, P, P, P, P, P,
                                ctypes.POINTER(Opts), P]


def amax(qkv, norm_wq, norm_wk, positions, *, heads: int, head_dim: int, rotary_dim: int,
         batch: int = 1, valid_len: int | None = None, n_axes: int | None = None, axis_dims=None,
         theta: float = 10000.0, eps: float = 1e-6, out=None, stream=None):
    """The amax pass alone (h3qk_amax): a float32 [3] CUDA tensor holding the
    largest |y| of Q, K and V over the valid rows."""
    import torch

    if qkv.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("qkv must be float16 or bfloat16")
    tokens = qkv.shape[0]
    seq = tokens // batch
    if valid_len is None:
        valid_len = seq
    if n_axes is None:
        n_axes = positions.shape[1] if positions is not None and positions.dim() == 2 else 3
    _need_common(qkv, norm_wq, norm_wk, positions, tokens=tokens, heads=heads, head_dim=head_dim,
                 rotary_dim=rotary_dim, n_axes=n_axes, batch=batch, valid_lens=None, device=qkv.device)
    if out is None:
        out = torch.empty(3, dtype=torch.float32, device=qkv.device)
    _need(out, "out", device=qkv.device, dtypes=(torch.float32,), min_numel=3)
    L = lib()
    _split_sigs(L)
    o = _opts_for(qkv, n_axes=n_axes, axis_dims=axis_dims, theta=theta, eps=eps, batch=batch)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(qkv.device):  # the library keys its caches on the current device
        st = int(L.h3qk_amax(qkv.data_ptr(), norm_wq.data_ptr(), norm_wk.data_ptr(), _ptr(positions), tokens,
                             heads, head_dim, rotary_dim, valid_len, out.data_ptr(), ctypes.byref(o), stream))
    if st != OK:
        raise H3QKError(st, status_string(st), int(L.h3qk_last_cuda_error()))
    return out


def cast(qkv, norm_wq, norm_wk, positions, amax_t, *, heads: int, head_dim: int, rotary_dim: int,
         batch: int = 1, valid_len: int | None = None, n_axes: int | None = None, axis_dims=None,
         theta: float = 10000.0, eps: float = 1e-6, out=None, out_scales=None, stream=None):
    """The cast pass alone (h3qk_cast) under dynamic scales derived from
    ``amax_t`` (float32 [3] CUDA tensor).  Returns (q, k, v, scales)."""
    import torch

    if qkv.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("qkv must be float16 or bfloat16")
    tokens = qkv.shape[0]
    seq = tokens // batch
    if valid_len is None:
        valid_len = seq
    if n_axes is None:
        n_axes = positions.shape[1] if positions is not None and positions.dim() == 2 else 3
    dev = qkv.device
    _need_common(qkv, norm_wq, norm_wk, positions, tokens=tokens, heads=heads, head_dim=head_dim,
                 rotary_dim=rotary_dim, n_axes=n_axes, batch=batch, valid_lens=None, device=dev)
    _need(amax_t, "amax_t", device=dev, dtypes=(torch.float32,), min_numel=3)
    shape = (batch, heads, seq, head_dim)
    if out is None:
        out = tuple(torch.empty(shape, dtype=torch.float8_e4m3fn, device=dev) for _ in range(3))
    if out_scales is None:
        out_scales = torch.empty(3, dtype=torch.float32, device=dev)
    q, k, v = out
    for t, name in zip((q, k, v), ("out[0]", "out[1]", "out[2]")):
        _need(t, name, device=dev, esz=1, numel=tokens * heads * head_dim)
    _need(out_scales, "out_scales", device=dev, dtypes=(torch.float32,), min_numel=3)
    L = lib()
    _split_sigs(L)
    o = _opts_for(qkv, n_axes=n_axes, axis_dims=axis_dims, theta=theta, eps=eps, batch=batch)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(qkv.device):  # the library keys its caches on the current device
        st = int(L.h3qk_cast(qkv.data_ptr(), norm_wq.data_ptr(), norm_wk.data_ptr(), _ptr(positions), tokens,
                             heads, head_dim, rotary_dim, valid_len, amax_t.data_ptr(), q.data_ptr(),
                             k.data_ptr(), v.data_ptr(), out_scales.data_ptr(), ctypes.byref(o), stream))
    if st != OK:
        raise H3QKError(st, status_string(st), int(L.h3qk_last_cuda_error()))
    return q, k, v, out_scales


def prepare_dynamic_sharded(qkv, norm_wq, norm_wk, positions, *, group=None, amax_fn=None,
                            cast_fn=None, **kw):
    """Dynamic e4m3 for rows sharded over the ranks of ``group``: the amax
    pass on this rank's rows, an all-reduce (MAX) of the three amax values
    over the group, then the cast pass with the shared scales, so every rank
    casts and dequantizes with the same descales.  With ``group`` None (one
    process) it equals prepare(..., scale_mode="dynamic").  ``amax_fn`` and
    ``cast_fn`` default to the library's passes (:func:`amax`, :func:`cast`)."""
    amax_fn = amax_fn or amax
    cast_fn = cast_fn or cast
    cast_kw = {k: v for k, v in kw.items()}
    amax_kw = {k: v for k, v in kw.items() if k not in ("out", "out_scales")}
    a = amax_fn(qkv, norm_wq, norm_wk, positions, **amax_kw)
    if group is not None:
        import torch.distributed as dist

        dist.all_reduce(a, op=dist.ReduceOp.MAX, group=group)
    return cast_fn(qkv, norm_wq, norm_wk, positions, a, **cast_kw)


def norm_rope_tensor(x, norm_w, positions, *, kind: str, heads: int, head_dim: int, rotary_dim: int,
                     batch: int = 1, valid_len: int | None = None, scale_mode: str = "none",
                     n_axes: int | None = None, axis_dims=None, theta: float = 10000.0, eps: float = 1e-6,
                     static_scale=None, out=None, out_scale=None, workspace=None, stream=None,
                     valid_lens=None, sat_counts=None):
    """One separately projected tensor x [tokens, >= heads*head_dim]
    (token-major [batch, S, heads, head_dim] rows): norm + RoPE for kind "q"
    or "k" (``norm_w`` float32 [head_dim]), identity for "v" (``norm_w`` may
    be None); 16-bit out (x's type) or e4m3 with its own descale.  Returns
    (out, scale): out token-major [batch, S, heads, head_dim], scale a
    float32 [1] tensor in e4m3 modes, else None."""
    import torch

    L = lib()
    fn = L.h3qk_norm_rope_tensor
    if fn.argtypes is None:
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        fn.restype = ctypes.c_int
        fn.argtypes = [P, P, P, I64, I32, I32, I32, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                       ctypes.POINTER(Opts), P]
    k = {"q": TENSOR_Q, "k": TENSOR_K, "v": TENSOR_V}[kind]
    if x.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("x must be float16 or bfloat16")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D [tokens, row_stride] with unit inner stride")
    tokens = x.shape[0]
    seq = tokens // batch
    if valid_len is None:
        valid_len = seq
    mode = _SCALE_NAMES[scale_mode]
    out_dt = (FP16 if x.dtype == torch.float16 else BF16) if mode == SCALE_NONE else E4M3
    if n_axes is None:
        n_axes = positions.shape[1] if positions is not None and positions.dim() == 2 else 3
    dev = x.device
    _need_rows(x, "x", heads * head_dim)
    if k != TENSOR_V:
        _need(norm_w, "norm_w", device=dev, dtypes=(torch.float32,), numel=head_dim)
        if positions is not None or rotary_dim > 0:
            _need(positions, "positions", device=dev, dtypes=(torch.int32,), numel=tokens * n_axes)
    _need(valid_lens, "valid_lens", device=dev, dtypes=(torch.int32,), numel=batch, optional=True)
    if out is None:
        tdt = x.dtype if out_dt != E4M3 else torch.float8_e4m3fn
        out = torch.empty((batch, seq, heads, head_dim), dtype=tdt, device=dev)
    _need(out, "out", device=dev, esz=1 if out_dt == E4M3 else 2, numel=tokens * heads * head_dim)
    if out_dt == E4M3 and out_scale is None:
        out_scale = torch.empty(1, dtype=torch.float32, device=dev)
    if out_dt == E4M3:
        _need(out_scale, "out_scale", device=dev, dtypes=(torch.float32,), min_numel=1)
    if mode == SCALE_STATIC:
        _need(static_scale, "static_scale", device=dev, dtypes=(torch.float32,), min_numel=1)
    _need(sat_counts, "sat_counts", device=dev, esz=4, min_numel=1, optional=True)
    if mode == SCALE_DYNAMIC and workspace is None:
        workspace = torch.empty(int(L.h3qk_workspace_bytes()) // 4, dtype=torch.int32, device=x.device)
    o = _opts_for(x, n_axes=n_axes, axis_dims=axis_dims, theta=theta, eps=eps, batch=batch)
    o.static_scales = _ptr(static_scale)
    o.valid_lens = _ptr(valid_lens)
    o.sat_counts = _ptr(sat_counts)
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(x.device):  # the library keys its caches on the current device
        st = int(fn(x.data_ptr(), _ptr(norm_w), _ptr(positions), tokens, heads, head_dim, rotary_dim, valid_len,
                    k, out_dt, mode, out.data_ptr(), _ptr(out_scale) if out_dt == E4M3 else None,
                    ctypes.byref(o), stream))
    if st != OK:
        raise H3QKError(st, status_string(st), int(L.h3qk_last_cuda_error()))
    return out, (out_scale if out_dt == E4M3 else None)


def silu_and_mul(x, *, out=None, stream=None):
    """SwiGLU after the w1 projection: x fp16/bf16 [rows, 2f] (gate | up,
    row stride a multiple of 8) -> out [rows, f] = silu(gate) * up, rounded
    as the library documents (h3qk_silu_and_mul)."""
    import torch

    L = lib()
    fn = L.h3qk_silu_and_mul
    if fn.argtypes is None:
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                       ctypes.c_void_p, ctypes.c_void_p]
    if x.dtype not in (torch.float16, torch.bfloat16) or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D fp16/bf16 tensor with unit inner stride")
    rows, two_f = x.shape
    f = two_f // 2
    if out is None:
        out = torch.empty((rows, f), dtype=x.dtype, device=x.device)
    _need(out, "out", device=x.device, esz=2, numel=rows * f)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    dt = FP16 if x.dtype == torch.float16 else BF16
    with torch.cuda.device(x.device):  # the library keys its caches on the current device
        st = int(fn(x.data_ptr(), dt, rows, f, x.stride(0), out.data_ptr(), stream))
    if st != OK:
        raise H3QKError(st, status_string(st), int(L.h3qk_last_cuda_error()))
    return out


def scaled_residual(residual, branch, scale, *, out=None, stream=None):
    """residual float32 [rows, C] + branch fp16/bf16 [rows, C] * scale float32
    [C] or [1], the product rounded on its own (h3qk_scaled_residual).
    ``out=residual`` updates in place."""
    import torch

    L = lib()
    fn = L.h3qk_scaled_residual
    if fn.argtypes is None:
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                       ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    if residual.dim() != 2:
        raise ValueError("residual must be 2-D [rows, C]")
    rows, C = residual.shape
    dev = residual.device
    _need(residual, "residual", device=dev, dtypes=(torch.float32,))
    _need(branch, "branch", device=dev, dtypes=(torch.float16, torch.bfloat16), numel=rows * C)
    if scale.numel() not in (1, C):
        raise ValueError(f"scale must have 1 or {C} elements, got {scale.numel()}")
    _need(scale, "scale", device=dev, dtypes=(torch.float32,))
    if out is None:
        out = torch.empty_like(residual)
    _need(out, "out", device=dev, dtypes=(torch.float32,), numel=rows * C)
    if stream is None:
        stream = torch.cuda.current_stream(residual.device).cuda_stream
    dt = FP16 if branch.dtype == torch.float16 else BF16
    with torch.cuda.device(residual.device):  # the library keys its caches on the current device
        st = int(fn(residual.data_ptr(), branch.data_ptr(), dt, scale.data_ptr(), rows, C, scale.numel(),
                    out.data_ptr(), stream))
    if st != OK:
        raise H3QKError(st, status_string(st), int(L.h3qk_last_cuda_error()))
    return out
