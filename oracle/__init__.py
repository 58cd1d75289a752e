"""CPU oracle of the fused QK-prep path (per-head RMSNorm of Q and K, partial
multi-axis RoPE, permute of the packed QKV projection to head-major Q/K/V,
optional per-tensor e4m3 cast with dynamic or static scales and a valid-prefix
mask).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the product library never does.  The
arithmetic lives in ``h3qk_oracle.c`` (plain C, one binary32 operation per
step, compiled with ``-ffp-contract=off``); this module only compiles it and
marshals numpy arrays through ctypes.  It imports nothing from the CUDA
package.

Every function of the C file cites the page passage it follows; the readings
taken where the pages are silent are marked "Reading:" there.

Parity status: each step is pinned by closed forms, invariants, brute force
and hand-worked values in ``tests/test_oracle_*.py``, and the whole path by
the rounding-point error bound of a float64 evaluation of the mathematics.
The pages print no numbers for this operation, so where they are silent (the
rounding points, the reduction order, the pair layout) the oracle follows the
readings marked "Reading:" in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h3qk_oracle.c")
_LIB = os.path.join(_HERE, "libh3qk_oracle.so")

FP16, BF16 = 1, 2
OUT_16B, OUT_E4M3 = 0, 1
SCALE_NONE, SCALE_DYNAMIC, SCALE_STATIC = 0, 1, 2
MAX_HD = 16384
MAX_PAIRS = 128

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libh3qk_oracle.so`` with gcc.  When
    H3QK_ORACLE_LIB names another build (the mutation test's broken copies),
    that file is loaded instead and nothing is compiled."""
    if os.environ.get("H3QK_ORACLE_LIB"):
        return os.environ["H3QK_ORACLE_LIB"]
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def source() -> str:
    """The C source of the library that ``lib()`` loads (a broken copy's own
    source when H3QK_ORACLE_LIB points at one)."""
    alt = os.environ.get("H3QK_ORACLE_LIB")
    if alt:
        cand = os.path.splitext(alt)[0] + ".c"
        if os.path.exists(cand):
            return cand
    return _SRC


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("seq", ctypes.c_int64),
        ("valid_len", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("n_axes", ctypes.c_int32),
        ("axis_dims", ctypes.c_int32 * 3),
        ("in_dtype", ctypes.c_int32),
        ("out_kind", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
        ("eps", ctypes.c_float),
        ("static_scales", ctypes.c_float * 3),
        ("theta", ctypes.c_double),
        ("out_layout", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("valid_lens", ctypes.c_void_p),
    ]


@dataclass
class Problem:
    """Sizes and options of one call.  ``axis_dims`` defaults to three equal
    even widths (t, h, w) when ``n_axes`` is 3, else ``(rotary_dim,)``."""

    batch: int
    seq: int
    heads: int
    head_dim: int
    rotary_dim: int
    n_axes: int = 3
    axis_dims: tuple = ()
    in_dtype: int = FP16
    out_kind: int = OUT_16B
    scale_mode: int = SCALE_NONE
    valid_len: int | None = None
    row_stride: int | None = None
    eps: float = 1e-6
    theta: float = 10000.0
    static_scales: tuple = (1.0, 1.0, 1.0)
    tensor: bool = False   # one [B, S, H, D] tensor instead of packed QKV rows
    out_layout: int = 0    # 0 head-major [B, H, S, D], 1 token-major [B, S, H, D]
    valid_lens: tuple | None = None  # per-item valid lengths (clamped to [0, S])

    def __post_init__(self):
        if not self.axis_dims:
            if self.n_axes == 3:
                self.axis_dims = (self.rotary_dim // 3,) * 3
            else:
                self.axis_dims = (self.rotary_dim,)
        if self.valid_len is None:
            self.valid_len = self.seq
        if self.row_stride is None:
            self.row_stride = (1 if self.tensor else 3) * self.heads * self.head_dim
        self.check()

    @property
    def rows(self) -> int:
        return self.batch * self.seq

    @property
    def hd(self) -> int:
        return self.heads * self.head_dim

    def check(self):
        D, R = self.head_dim, self.rotary_dim
        if D % 8 or not (8 <= D <= 256):
            raise ValueError("head_dim must be a multiple of 8 in [8, 256]")
        if R % 2 or R > D or R // 2 > MAX_PAIRS:
            raise ValueError("rotary_dim must be even and <= head_dim")
        if len(self.axis_dims) != self.n_axes or sum(self.axis_dims) != R:
            raise ValueError("axis_dims must have n_axes entries summing to rotary_dim")
        if any(d % 2 for d in self.axis_dims):
            raise ValueError("axis widths must be even")
        if self.hd > MAX_HD:
            raise ValueError("heads * head_dim too large for the oracle")
        if not (0 <= self.valid_len <= self.seq):
            raise ValueError("valid_len must lie in [0, seq]")
        if self.row_stride < (1 if self.tensor else 3) * self.hd:
            raise ValueError("row_stride shorter than a row")

    def c(self) -> _Problem:
        p = _Problem()
        p.batch, p.seq, p.valid_len, p.row_stride = self.batch, self.seq, self.valid_len, self.row_stride
        p.heads, p.head_dim, p.rotary_dim, p.n_axes = self.heads, self.head_dim, self.rotary_dim, self.n_axes
        dims = list(self.axis_dims) + [0] * (3 - len(self.axis_dims))
        p.axis_dims = (ctypes.c_int32 * 3)(*dims)
        p.in_dtype, p.out_kind, p.scale_mode = self.in_dtype, self.out_kind, self.scale_mode
        p.eps = self.eps
        p.static_scales = (ctypes.c_float * 3)(*[float(s) for s in self.static_scales])
        p.theta = self.theta
        p.out_layout = self.out_layout
        if self.valid_lens is not None:
            self._vl = np.ascontiguousarray(self.valid_lens, np.int32)
            assert self._vl.shape == (self.batch,)
            p.valid_lens = self._vl.ctypes.data
        return p


_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            PP = ctypes.POINTER(_Problem)
            sigs = {
                "h3o_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
                "h3o_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "h3o_f32_to_e4m3": (ctypes.c_uint8, [ctypes.c_float]),
                "h3o_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "h3o_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "h3o_e4m3_to_f32": (ctypes.c_float, [ctypes.c_uint8]),
                "h3o_f32_to_f16_array": (None, [_P, _P, _I64]),
                "h3o_f32_to_bf16_array": (None, [_P, _P, _I64]),
                "h3o_f32_to_e4m3_array": (None, [_P, _P, _I64]),
                "h3o_sincos_array": (None, [_P, _P, _P, _I64]),
                "h3o_inv_freq": (None, [ctypes.c_double, ctypes.c_int, _P]),
                "h3o_sumsq": (ctypes.c_float, [_P, ctypes.c_int]),
                "h3o_rms_inv": (ctypes.c_float, [_P, ctypes.c_int, ctypes.c_float]),
                "h3o_norm_head": (None, [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_float, _P]),
                "h3o_rotate_pair": (None, [ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_uint16, ctypes.c_uint16, _P, _P]),
                "h3o_row16": (None, [PP, _P, _P, _P, _P, _I64, _P, _P, _P]),
                "h3o_prepare16_rows": (None, [PP, _P, _P, _P, _P, _I64, _I64, _P, _P, _P]),
                "h3o_amax_rows": (None, [PP, _P, _P, _P, _P, _I64, _I64, _P]),
                "h3o_scales": (None, [PP, _P, _P, _P]),
                "h3o_cast_rows": (None, [PP, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P]),
                "h3o_cast_row": (None, [PP, _P, _P, _P, _P, _I64, _P, _P, _P, _P]),
                "h3o_prepare": (None, [PP, _P, _P, _P, _P, _P, _P, _P, _P]),
                "h3o_angles_array": (None, [PP, _P, _I64, _P]),
                "h3o_sat_rows": (None, [PP, _P, _P, _P, _P, _I64, _I64, _P, _P]),
                "h3o_exp": (ctypes.c_float, [ctypes.c_float]),
                "h3o_silu": (ctypes.c_float, [ctypes.c_float]),
                "h3o_exp_array": (None, [_P, _P, _I64]),
                "h3o_silu_and_mul_rows": (None, [ctypes.c_int, _P, _I64, ctypes.c_int, _I64, _P]),
                "h3o_scaled_residual": (None, [ctypes.c_int, _P, _P, _P, _I64, ctypes.c_int, ctypes.c_int, _P]),
                "h3o_tensor_row16": (None, [PP, ctypes.c_int, _P, _P, _P, _I64, _P]),
                "h3o_tensor16_rows": (None, [PP, ctypes.c_int, _P, _P, _P, _I64, _I64, _P]),
                "h3o_tensor_amax_rows": (ctypes.c_float, [PP, ctypes.c_int, _P, _P, _P, _I64, _I64]),
                "h3o_tensor_cast_rows": (None, [PP, ctypes.c_int, _P, _P, _P, _I64, _I64, ctypes.c_float, _P]),
                "h3o_problem_inv_freq_public": (None, [PP, _P]),
                "h3o_norm_head_f32": (None, [_P, _P, ctypes.c_int, ctypes.c_float, _P]),
                "h3o_rotate_f32": (None, [ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                          _P, _P]),
                "h3o_sage_rows": (None, [PP, _P, _P, _P, _P, ctypes.c_float, _I64, _I64, _P, _P, _P]),
            }
            for name, (res, args) in sigs.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Scalar / element-wise steps (for the pins).
# --------------------------------------------------------------------------

def f32_to_f16(x) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    y = np.empty(x.shape, np.uint16)
    lib().h3o_f32_to_f16_array(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_bf16(x) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    y = np.empty(x.shape, np.uint16)
    lib().h3o_f32_to_bf16_array(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_e4m3(x) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    y = np.empty(x.shape, np.uint8)
    lib().h3o_f32_to_e4m3_array(_ptr(x), _ptr(y), x.size)
    return y


def sincos(a):
    a = _c(a, np.float32).reshape(-1)
    s = np.empty_like(a)
    c = np.empty_like(a)
    lib().h3o_sincos_array(_ptr(a), _ptr(s), _ptr(c), a.size)
    return s, c


def inv_freq(theta: float, d: int) -> np.ndarray:
    out = np.empty(d // 2, np.float32)
    lib().h3o_inv_freq(float(theta), int(d), _ptr(out))
    return out


def sumsq(x) -> np.float32:
    x = _c(x, np.float32)
    return np.float32(lib().h3o_sumsq(_ptr(x), x.size))


def rms_inv(x, eps: float = 1e-6) -> np.float32:
    x = _c(x, np.float32)
    return np.float32(lib().h3o_rms_inv(_ptr(x), x.size, eps))


def norm_head(x, w, dtype: int = FP16, eps: float = 1e-6) -> np.ndarray:
    """x: float32 [D] (already 16-bit-representable), w: float32 [D] -> 16-bit codes."""
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    n = np.empty(x.size, np.uint16)
    lib().h3o_norm_head(dtype, _ptr(x), _ptr(w), x.size, eps, _ptr(n))
    return n


def rotate_pair(c: float, s: float, u16: int, v16: int, dtype: int = FP16):
    uo = np.zeros(1, np.uint16)
    vo = np.zeros(1, np.uint16)
    lib().h3o_rotate_pair(dtype, float(c), float(s), int(u16), int(v16), _ptr(uo), _ptr(vo))
    return int(uo[0]), int(vo[0])


def angles(pb: Problem, pos: np.ndarray) -> np.ndarray:
    pos = _c(pos, np.int32).reshape(-1, pb.n_axes)
    out = np.empty((pos.shape[0], pb.rotary_dim // 2), np.float32)
    lib().h3o_angles_array(ctypes.byref(pb.c()), _ptr(pos), pos.shape[0], _ptr(out))
    return out


def problem_inv_freq(pb: Problem) -> np.ndarray:
    out = np.empty(max(pb.rotary_dim // 2, 1), np.float32)
    lib().h3o_problem_inv_freq_public(ctypes.byref(pb.c()), _ptr(out))
    return out[: pb.rotary_dim // 2]


# --------------------------------------------------------------------------
# The path.
# --------------------------------------------------------------------------

def _inputs(pb: Problem, qkv, wq, wk, pos):
    qkv = _c(qkv, np.uint16)
    if qkv.ndim != 2 or qkv.shape[0] != pb.rows or qkv.shape[1] != pb.row_stride:
        raise ValueError(f"qkv must be uint16 [{pb.rows}, {pb.row_stride}]")
    wq = _c(wq, np.float32)
    wk = _c(wk, np.float32)
    if wq.shape != (pb.head_dim,) or wk.shape != (pb.head_dim,):
        raise ValueError("norm weights must be float32 [head_dim]")
    pos = _c(pos, np.int32)
    if pos.shape != (pb.rows, pb.n_axes):
        raise ValueError(f"positions must be int32 [{pb.rows}, {pb.n_axes}]")
    return qkv, wq, wk, pos


def row16(pb: Problem, qkv, wq, wk, pos, rows):
    """16-bit Q, K, V of the given rows: three uint16 arrays [len(rows), H, D]."""
    qkv, wq, wk, pos = _inputs(pb, qkv, wq, wk, pos)
    rows = np.asarray(rows, np.int64).reshape(-1)
    out = [np.empty((rows.size, pb.heads, pb.head_dim), np.uint16) for _ in range(3)]
    L, cp = lib(), pb.c()
    for i, r in enumerate(rows):
        L.h3o_row16(ctypes.byref(cp), _ptr(qkv), _ptr(wq), _ptr(wk), _ptr(pos), int(r),
                    _ptr(out[0][i]), _ptr(out[1][i]), _ptr(out[2][i]))
    return tuple(out)


def _ranges(n: int, parts: int):
    parts = max(1, min(parts, n)) if n else 1
    step = -(-n // parts) if n else 0
    return [(i, min(n, i + step)) for i in range(0, n, step)] if n else []


def amax(pb: Problem, qkv, wq, wk, pos, threads: int = 1, rows: tuple | None = None) -> np.ndarray:
    """Per-tensor amax over the valid rows (of ``rows=(r0, r1)`` if given),
    split over ``threads`` row ranges (max is order-independent)."""
    qkv, wq, wk, pos = _inputs(pb, qkv, wq, wk, pos)
    r0, r1 = rows if rows is not None else (0, pb.rows)
    cp = pb.c()
    L = lib()

    def one(rg):
        m = np.zeros(3, np.float32)
        L.h3o_amax_rows(ctypes.byref(cp), _ptr(qkv), _ptr(wq), _ptr(wk), _ptr(pos),
                        r0 + rg[0], r0 + rg[1], _ptr(m))
        return m

    parts = _ranges(r1 - r0, threads)
    if not parts:
        return np.zeros(3, np.float32)
    if threads <= 1:
        ms = [one(rg) for rg in parts]
    else:
        with ThreadPoolExecutor(threads) as ex:
            ms = list(ex.map(one, parts))
    return np.max(np.stack(ms), axis=0).astype(np.float32)


def scales(pb: Problem, amax_vals) -> tuple[np.ndarray, np.ndarray]:
    a = _c(amax_vals, np.float32)
    s = np.empty(3, np.float32)
    i = np.empty(3, np.float32)
    lib().h3o_scales(ctypes.byref(pb.c()), _ptr(a), _ptr(s), _ptr(i))
    return s, i


def prepare(pb: Problem, qkv, wq, wk, pos, out=None, threads: int = 1):
    """The whole path.  Returns (q, k, v, scales): head-major [B, H, S, D]
    uint16 codes (16-bit mode) or uint8 e4m3 codes, and the three descales
    (None in 16-bit mode).  Rows past valid_len keep the contents of ``out``
    (zeros when ``out`` is None)."""
    qkv, wq, wk, pos = _inputs(pb, qkv, wq, wk, pos)
    shape = ((pb.batch, pb.seq, pb.heads, pb.head_dim) if pb.out_layout == 1
             else (pb.batch, pb.heads, pb.seq, pb.head_dim))
    odt = np.uint16 if pb.out_kind == OUT_16B else np.uint8
    if out is None:
        out = tuple(np.zeros(shape, odt) for _ in range(3))
    q, k, v = out
    for t in out:
        assert t.dtype == odt and t.shape == shape and t.flags.c_contiguous
    L, cp = lib(), pb.c()
    args = (ctypes.byref(cp), _ptr(qkv), _ptr(wq), _ptr(wk), _ptr(pos))
    if threads <= 1:
        sc = np.zeros(3, np.float32)
        L.h3o_prepare(*args, _ptr(q), _ptr(k), _ptr(v), _ptr(sc))
        return q, k, v, (sc if pb.out_kind == OUT_E4M3 else None)
    parts = _ranges(pb.rows, threads)
    with ThreadPoolExecutor(threads) as ex:
        if pb.out_kind == OUT_16B:
            list(ex.map(lambda rg: L.h3o_prepare16_rows(*args, rg[0], rg[1], _ptr(q), _ptr(k), _ptr(v)),
                        parts))
            return q, k, v, None
        am = np.zeros(3, np.float32)
        if pb.scale_mode == SCALE_DYNAMIC:
            am = amax(pb, qkv, wq, wk, pos, threads=threads)
        sc, inv = scales(pb, am)
        list(ex.map(lambda rg: L.h3o_cast_rows(*args, rg[0], rg[1], _ptr(inv), _ptr(q), _ptr(k), _ptr(v)),
                    parts))
    return q, k, v, sc


def sage(pb: Problem, qkv, wq, wk, pos, kv_scale: float = 1.0, out=None, threads: int = 1):
    """The sage-attention outputs: (q, k, v) head-major [B, H, S, D] (or
    token-major, ``pb.out_layout``); q and k float32 (k times kv_scale), v
    binary16 codes (uint16) of v times kv_scale.  Rows past the valid prefix
    keep the contents of ``out`` (zeros when None)."""
    qkv, wq, wk, pos = _inputs(pb, qkv, wq, wk, pos)
    shape = ((pb.batch, pb.seq, pb.heads, pb.head_dim) if pb.out_layout == 1
             else (pb.batch, pb.heads, pb.seq, pb.head_dim))
    if out is None:
        out = (np.zeros(shape, np.float32), np.zeros(shape, np.float32), np.zeros(shape, np.uint16))
    q, k, v = out
    for t, dt in zip(out, (np.float32, np.float32, np.uint16)):
        assert t.dtype == dt and t.shape == shape and t.flags.c_contiguous
    L, cp = lib(), pb.c()
    args = (ctypes.byref(cp), _ptr(qkv), _ptr(wq), _ptr(wk), _ptr(pos), float(kv_scale))
    parts = _ranges(pb.rows, max(1, threads))
    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(lambda rg: L.h3o_sage_rows(*args, rg[0], rg[1], _ptr(q), _ptr(k), _ptr(v)), parts))
    return q, k, v


def norm_head_f32(x, w, eps: float = 1e-6) -> np.ndarray:
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    y = np.empty(x.size, np.float32)
    lib().h3o_norm_head_f32(_ptr(x), _ptr(w), x.size, eps, _ptr(y))
    return y


def rotate_f32(c: float, s: float, u: float, v: float):
    uo = np.empty(1, np.float32)
    vo = np.empty(1, np.float32)
    lib().h3o_rotate_f32(float(c), float(s), float(u), float(v), _ptr(uo), _ptr(vo))
    return uo[0], vo[0]


def cast_rows(pb: Problem, qkv, wq, wk, pos, inv, rows):
    """e4m3 codes of the given rows under the factors ``inv``: three uint8
    arrays [len(rows), H, D] (rows taken as valid)."""
    qkv, wq, wk, pos = _inputs(pb, qkv, wq, wk, pos)
    inv = _c(inv, np.float32)
    rows = np.asarray(rows, np.int64).reshape(-1)
    out = [np.empty((rows.size, pb.heads, pb.head_dim), np.uint8) for _ in range(3)]
    L, cp = lib(), pb.c()
    for i, r in enumerate(rows):
        L.h3o_cast_row(ctypes.byref(cp), _ptr(qkv), _ptr(wq), _ptr(wk), _ptr(pos), int(r), _ptr(inv),
                       _ptr(out[0][i]), _ptr(out[1][i]), _ptr(out[2][i]))
    return tuple(out)


def f16_to_f32(codes) -> np.ndarray:
    """16-bit IEEE codes -> float32 (numpy's own conversion, exact)."""
    return np.asarray(codes, np.uint16).view(np.float16).astype(np.float32)


def bf16_to_f32(codes) -> np.ndarray:
    """bfloat16 codes -> float32 (exact: the codes are the upper 16 bits)."""
    return (np.asarray(codes, np.uint32) << 16).astype(np.uint32).view(np.float32)


# --------------------------------------------------------------------------
# The single-tensor variant: one [B, S, H, D] tensor, norm + RoPE (kind 0 Q,
# 1 K) or identity (kind 2 V), token-major output.
# --------------------------------------------------------------------------

def tensor_prepare(pb: Problem, kind: int, x, w, pos, out=None, threads: int = 1):
    """Returns (out, scale): token-major [B, S, H, D] uint16 codes (16-bit
    mode) or uint8 e4m3 codes and the one descale (None in 16-bit mode).
    Rows past valid_len keep the contents of ``out``."""
    assert pb.tensor, "tensor_prepare needs Problem(tensor=True)"
    x = _c(x, np.uint16)
    if x.ndim != 2 or x.shape != (pb.rows, pb.row_stride):
        raise ValueError(f"x must be uint16 [{pb.rows}, {pb.row_stride}]")
    w = _c(w if w is not None else np.zeros(pb.head_dim, np.float32), np.float32)
    pos = _c(pos, np.int32)
    shape = (pb.batch, pb.seq, pb.heads, pb.head_dim)
    odt = np.uint16 if pb.out_kind == OUT_16B else np.uint8
    if out is None:
        out = np.zeros(shape, odt)
    assert out.dtype == odt and out.shape == shape and out.flags.c_contiguous
    L, cp = lib(), pb.c()
    args = (ctypes.byref(cp), int(kind), _ptr(x), _ptr(w), _ptr(pos))
    parts = _ranges(pb.rows, threads)
    with ThreadPoolExecutor(max(1, threads)) as ex:
        if pb.out_kind == OUT_16B:
            list(ex.map(lambda rg: L.h3o_tensor16_rows(*args, rg[0], rg[1], _ptr(out)), parts))
            return out, None
        am = 0.0
        if pb.scale_mode == SCALE_DYNAMIC:
            am = max([0.0] + list(ex.map(lambda rg: L.h3o_tensor_amax_rows(*args, rg[0], rg[1]), parts)))
        sc, inv = scales(pb, np.array([am, am, am], np.float32))
        scale, factor = float(sc[0]), float(inv[0])
        list(ex.map(lambda rg: L.h3o_tensor_cast_rows(*args, rg[0], rg[1], factor, _ptr(out)), parts))
    return out, np.float32(scale)


def sat_counts(pb: Problem, qkv, wq, wk, pos, inv) -> np.ndarray:
    """Per-tensor counts of valid-row values whose scaled magnitude exceeds
    448 under the factors ``inv``."""
    qkv, wq, wk, pos = _inputs(pb, qkv, wq, wk, pos)
    inv = _c(inv, np.float32)
    counts = np.zeros(3, np.uint32)
    lib().h3o_sat_rows(ctypes.byref(pb.c()), _ptr(qkv), _ptr(wq), _ptr(wk), _ptr(pos), 0, pb.rows,
                       _ptr(inv), _ptr(counts))
    return counts


# --------------------------------------------------------------------------
# Adjacent VAE-block operations (SwiGLU, scaled residual).
# --------------------------------------------------------------------------

def exp(x) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    y = np.empty_like(x)
    lib().h3o_exp_array(_ptr(x), _ptr(y), x.size)
    return y


def silu_and_mul(x, f: int, dtype: int = FP16) -> np.ndarray:
    """x: uint16 codes [rows, >= 2f] (gate | up); returns uint16 [rows, f]."""
    x = _c(x, np.uint16)
    rows = x.shape[0]
    out = np.empty((rows, f), np.uint16)
    lib().h3o_silu_and_mul_rows(dtype, _ptr(x), rows, f, x.shape[1], _ptr(out))
    return out


def scaled_residual(residual, branch, scale, dtype: int = FP16) -> np.ndarray:
    """residual float32 [rows, C], branch uint16 codes [rows, C], scale
    float32 [C] or [1]; returns float32 [rows, C]."""
    residual = _c(residual, np.float32)
    branch = _c(branch, np.uint16)
    scale = _c(scale, np.float32).reshape(-1)
    rows, C = residual.shape
    assert branch.shape == (rows, C) and scale.size in (1, C)
    out = np.empty_like(residual)
    lib().h3o_scaled_residual(dtype, _ptr(residual), _ptr(branch), _ptr(scale), rows, C, scale.size, _ptr(out))
    return out
