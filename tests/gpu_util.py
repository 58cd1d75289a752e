"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding on the seeded inputs, run the CPU oracle on the same inputs, compare
bytes."""
from __future__ import annotations

import os

import numpy as np

import oracle
from video_vae_decoder_qkv_gb300 import workloads as W

THREADS = max(1, min(32, os.cpu_count() or 1))


def problem(spec: W.Spec, **kw) -> oracle.Problem:
    d = dict(batch=spec.batch, seq=spec.seq, heads=spec.heads, head_dim=spec.head_dim,
             rotary_dim=spec.rotary_dim, n_axes=spec.n_axes, axis_dims=tuple(spec.axis_dims),
             in_dtype=spec.in_dtype, out_kind=spec.out_kind, scale_mode=spec.scale_mode,
             valid_len=spec.valid_len, row_stride=spec.row_stride, eps=spec.eps, theta=spec.theta)
    d.update(kw)
    return oracle.Problem(**d)


def _input_key(spec: W.Spec):
    d = dict(spec.__dict__)
    for k in ("name", "out_kind", "scale_mode", "valid_len"):
        d.pop(k)
    return tuple(sorted((k, str(v)) for k, v in d.items()))


_CACHE: dict = {}


def inputs(spec: W.Spec) -> W.Inputs:
    """Seeded inputs, reused across tests for specs that share them."""
    key = _input_key(spec)
    if key not in _CACHE:
        if len(_CACHE) >= 2:
            _CACHE.pop(next(iter(_CACHE)))
        _CACHE[key] = W.generate(spec)
    inp = _CACHE[key]
    return W.Inputs(spec, inp.qkv, inp.wq, inp.wk, inp.pos, inp.static_scales, inp.outlier_cols)


def to_device(inp: W.Inputs):
    import torch

    dt = torch.float16 if inp.spec.in_dtype == W.FP16 else torch.bfloat16
    qkv = torch.from_numpy(inp.qkv.view(np.int16)).cuda().view(dt)
    wq = torch.from_numpy(inp.wq).cuda()
    wk = torch.from_numpy(inp.wk).cuda()
    pos = torch.from_numpy(inp.pos).cuda()
    return qkv, wq, wk, pos


def out_tensors(spec: W.Spec, fill: int | None = None):
    import torch

    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    if spec.out_kind == W.OUT_E4M3:
        t = [torch.empty(shape, dtype=torch.uint8, device="cuda") for _ in range(3)]
        if fill is not None:
            for x in t:
                x.fill_(fill & 0xFF)
        return tuple(x.view(torch.float8_e4m3fn) for x in t)
    dt = torch.float16 if spec.in_dtype == W.FP16 else torch.bfloat16
    t = [torch.empty(shape, dtype=torch.int16, device="cuda") for _ in range(3)]
    if fill is not None:
        f = fill & 0xFFFF
        for x in t:
            x.fill_(f - 0x10000 if f >= 0x8000 else f)
    return tuple(x.view(dt) for x in t)


def gpu_prepare(inp: W.Inputs, fill: int | None = None, static=None, dev=None, **kw):
    """Run the CUDA path; returns device tensors (q, k, v, scales)."""
    import torch

    from video_vae_decoder_qkv_gb300 import prepare

    spec = inp.spec
    qkv, wq, wk, pos = dev if dev is not None else to_device(inp)
    mode = {W.SCALE_NONE: "none", W.SCALE_DYNAMIC: "dynamic", W.SCALE_STATIC: "static"}[spec.scale_mode]
    st = None
    if spec.scale_mode == W.SCALE_STATIC:
        st = torch.from_numpy(np.asarray(static if static is not None else inp.static_scales,
                                         np.float32)).cuda()
    out = out_tensors(spec, fill)
    q, k, v, sc = prepare(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim,
                          rotary_dim=spec.rotary_dim, batch=spec.batch, valid_len=spec.valid_len,
                          scale_mode=mode, n_axes=spec.n_axes, axis_dims=spec.axis_dims,
                          theta=spec.theta, eps=spec.eps, static_scales=st, out=out, **kw)
    return q, k, v, sc


def as_codes(t):
    """The same storage as integer codes (uint8 for e4m3, int16 for 16-bit)."""
    import torch

    return t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)


def host_codes(t) -> np.ndarray:
    import torch

    if t.element_size() == 1:
        return t.view(torch.uint8).cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_full(inp: W.Inputs, static=None, fill: int | None = None):
    """The oracle's whole-path outputs (threads over row ranges)."""
    spec = inp.spec
    kw = {}
    if spec.scale_mode == W.SCALE_STATIC:
        kw["static_scales"] = tuple(float(x) for x in (static if static is not None else inp.static_scales))
    pb = problem(spec, **kw)
    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    odt = np.uint8 if spec.out_kind == W.OUT_E4M3 else np.uint16
    out = None
    if fill is not None:
        out = tuple(np.full(shape, fill, odt) for _ in range(3))
    return oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos, out=out, threads=THREADS)


def _nan_mask(codes: np.ndarray, kind: str) -> np.ndarray:
    if kind == "f32":
        c = codes.astype(np.uint32)
        return ((c & 0x7F800000) == 0x7F800000) & ((c & 0x7FFFFF) != 0)
    if kind == "e4m3":
        return (codes & 0x7F) == 0x7F
    if kind == "fp16":
        return ((codes & 0x7C00) == 0x7C00) & ((codes & 0x3FF) != 0)
    return ((codes & 0x7F80) == 0x7F80) & ((codes & 0x7F) != 0)


def assert_codes_equal(got: np.ndarray, want: np.ndarray, what: str, nan_kind: str | None = None):
    """Bit-exact comparison; with ``nan_kind`` ("fp16", "bf16", "e4m3") any
    NaN code matches any NaN code at the same position."""
    if nan_kind is not None:
        gn, wn = _nan_mask(got, nan_kind), _nan_mask(want, nan_kind)
        assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
        got = np.where(gn, 0, got)
        want = np.where(wn, 0, want)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} codes differ; first at {i}: "
                             f"gpu {int(got[i]):#x} oracle {int(want[i]):#x}")
