"""Seeded synthetic inputs for the fused QK-prep path.

This module only draws inputs; it holds none of the path's arithmetic.  The
tests feed the same arrays to the CPU oracle and to the CUDA library, and the
benchmark times the CUDA library on them.

The five named workloads follow the shapes of the MiniMax-H3 pages:
- ``tiny``: a 2x4x6 token grid, 4 heads of 64, parity only;
- ``decoder_tile``: one 288x272-pixel decoder tile at 16 px per token, a
  16x18x17 token grid (TensorRT-LLM #21484 "FP8 tiled VAE decoder and a
  leaner pipeline schedule", Summary: tiles of 288x272);
- ``batched_fp8``: 8 such tiles in one call with the dynamic per-tensor e4m3
  cast (TensorRT-LLM #21485 "cuDNN FP8 attention path for MiniMax-H3 on SM107
  under Ulysses", Summary bullet 2);
- ``latent_65k``: the untiled 544x960 latent grid, 32x34x60 = 65,280 tokens,
  24 heads of 128;
- ``prefix_104k``: 104,076 valid rows padded to 104,080, a multiple of 8, as
  the Ulysses padding of the same TensorRT-LLM #21485 Summary bullet 1,
  with 1-D positions and 40 heads of 128.

Value recipe (every workload): the packed QKV projection is drawn ~N(0, 1)
in float32 and rounded to the 16-bit input type; a fixed set of
ceil(frac * 3*H*D) outlier columns, drawn once, is multiplied by a factor in
every row before rounding; the norm weights are ~U(0.5, 1.5); static e4m3
descales ~U(0.01, 0.1).  Positions are tile-local (t, h, w) grid indices of
token n = (t*Hg + h)*Wg + w, or 0..S-1 for 1-D positions.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

FP16, BF16 = 1, 2
OUT_16B, OUT_E4M3 = 0, 1
SCALE_NONE, SCALE_DYNAMIC, SCALE_STATIC = 0, 1, 2

_CHUNK_ROWS = 2048


@dataclass
class Spec:
    """Sizes, options and value recipe of one synthetic workload."""

    name: str
    batch: int
    seq: int
    heads: int
    head_dim: int
    rotary_dim: int
    grid: tuple | None = None          # (T, Hg, Wg) for 3-axis positions
    n_axes: int = 3
    axis_dims: tuple = ()
    in_dtype: int = FP16
    out_kind: int = OUT_16B
    scale_mode: int = SCALE_NONE
    valid_len: int | None = None
    row_stride: int | None = None
    eps: float = 1e-6
    theta: float = 10000.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    dist: str = "normal"               # normal | zeros | huge | tiny | subsq | unique
    seed: int = 0

    def __post_init__(self):
        if not self.axis_dims:
            self.axis_dims = ((self.rotary_dim // 3,) * 3 if self.n_axes == 3
                              else (self.rotary_dim,))
        if self.valid_len is None:
            self.valid_len = self.seq
        if self.row_stride is None:
            self.row_stride = 3 * self.heads * self.head_dim

    @property
    def rows(self) -> int:
        return self.batch * self.seq

    @property
    def hd(self) -> int:
        return self.heads * self.head_dim

    def with_(self, **kw) -> "Spec":
        d = dict(self.__dict__)
        d.update(kw)
        if "rotary_dim" in kw or "n_axes" in kw:
            d.setdefault("axis_dims", ())
            if "axis_dims" not in kw:
                d["axis_dims"] = ()
        if "seq" in kw and "valid_len" not in kw:
            d["valid_len"] = None
        if ("heads" in kw or "head_dim" in kw) and "row_stride" not in kw:
            d["row_stride"] = None
        return Spec(**d)

    def valid_rows(self) -> int:
        return self.batch * self.valid_len

    def algorithmic_bytes(self) -> int:
        """Bytes the path must move over the valid rows: the input read once
        per pass (twice for the dynamic cast) and the outputs written once."""
        n = self.valid_rows() * self.hd
        if self.out_kind == OUT_16B:
            return 12 * n
        return (15 if self.scale_mode == SCALE_DYNAMIC else 9) * n


@dataclass
class Inputs:
    spec: Spec
    qkv: np.ndarray            # uint16 codes [rows, row_stride]
    wq: np.ndarray             # float32 [D]
    wk: np.ndarray             # float32 [D]
    pos: np.ndarray            # int32 [rows, n_axes]
    static_scales: np.ndarray  # float32 [3]
    outlier_cols: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))


def _to16(x: np.ndarray, dtype: int) -> np.ndarray:
    """float32 values -> 16-bit codes, with numpy's (fp16) or torch's (bf16)
    round-to-nearest-even conversion."""
    if dtype == FP16:
        return x.astype(np.float16).view(np.uint16)
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def positions(spec: Spec) -> np.ndarray:
    """Tile-local positions of every row, int32 [rows, n_axes]."""
    s = np.arange(spec.seq, dtype=np.int64)
    if spec.n_axes == 3:
        if spec.grid is not None:
            T, Hg, Wg = spec.grid
            assert T * Hg * Wg == spec.seq, "grid must cover the sequence"
        else:
            Hg, Wg = 1, spec.seq
        p = np.stack([s // (Hg * Wg), (s // Wg) % Hg, s % Wg], axis=1)
    else:
        p = s[:, None]
    p = np.tile(p, (spec.batch, 1))
    return np.ascontiguousarray(p, dtype=np.int32)


def generate(spec: Spec) -> Inputs:
    """Draw the inputs of ``spec`` (deterministic in ``spec.seed``)."""
    head = np.random.default_rng([spec.seed, 0])
    ncols = 3 * spec.hd
    n_out = math.ceil(spec.outlier_frac * ncols) if spec.outlier_frac > 0 else 0
    cols = np.sort(head.choice(ncols, size=n_out, replace=False)) if n_out else np.zeros(0, np.int64)
    wq = head.uniform(0.5, 1.5, spec.head_dim).astype(np.float32)
    wk = head.uniform(0.5, 1.5, spec.head_dim).astype(np.float32)
    static = head.uniform(0.01, 0.1, 3).astype(np.float32)

    qkv = np.zeros((spec.rows, spec.row_stride), np.uint16)

    def fill(c0: int) -> None:
        # each chunk has its own seed, so chunks may be drawn in any order
        c1 = min(spec.rows, c0 + _CHUNK_ROWS)
        rng = np.random.default_rng([spec.seed, 1, c0 // _CHUNK_ROWS])
        n = c1 - c0
        if spec.dist == "unique":
            # every element a distinct finite code (layout checks); squares stay finite
            idx = (np.arange(c0, c1, dtype=np.int64)[:, None] * ncols
                   + np.arange(ncols, dtype=np.int64)[None, :])
            top = 0x7BFF if spec.in_dtype == FP16 else 0x46FF
            qkv[c0:c1, :ncols] = (idx % top + 1).astype(np.uint16)
            return
        if spec.dist == "normal":
            x = rng.standard_normal((n, ncols), dtype=np.float32)
        elif spec.dist == "zeros":
            x = np.zeros((n, ncols), np.float32)
        elif spec.dist == "huge":
            # large magnitudes that push the 16-bit and e4m3 ranges
            mag = 60000.0 if spec.in_dtype == FP16 else 1e18
            x = (rng.uniform(-1, 1, (n, ncols)) * mag).astype(np.float32)
        elif spec.dist == "subsq":
            # magnitudes whose squares are not exact in binary32 (bf16 values
            # in [2^-80, 2^-62]; fp16 values at its smallest subnormals)
            lo, hi = (-80.0, -62.0) if spec.in_dtype == BF16 else (-24.0, -20.0)
            mag = np.exp2(rng.uniform(lo, hi, (n, ncols)))
            x = (np.where(rng.random((n, ncols)) < 0.5, -mag, mag)).astype(np.float32)
        elif spec.dist == "tiny":
            # magnitudes around the 16-bit subnormal range
            lo = 2.0 ** -24 if spec.in_dtype == FP16 else 2.0 ** -133
            x = (rng.uniform(-64, 64, (n, ncols)) * lo).astype(np.float32)
        else:
            raise ValueError(spec.dist)
        if n_out:
            x[:, cols] *= np.float32(spec.outlier_scale)
        if spec.dist == "huge":
            # keep every input finite in the 16-bit type (non-finite inputs are
            # a separate case)
            top = 65504.0 if spec.in_dtype == FP16 else 3.3895313e38
            np.clip(x, -top, top, out=x)
        qkv[c0:c1, :ncols] = _to16(x, spec.in_dtype)

    starts = list(range(0, spec.rows, _CHUNK_ROWS))
    if len(starts) > 2:
        workers = max(1, min(16, os.cpu_count() or 1))
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, starts))
    else:
        for c0 in starts:
            fill(c0)
    return Inputs(spec, qkv, wq, wk, positions(spec), static, cols)


TINY = Spec("tiny", batch=1, seq=48, heads=4, head_dim=64, rotary_dim=48, grid=(2, 4, 6),
            in_dtype=FP16, seed=0)
DECODER_TILE = Spec("decoder_tile", batch=1, seq=4896, heads=16, head_dim=64, rotary_dim=48,
                    grid=(16, 18, 17), in_dtype=FP16, outlier_frac=0.001, outlier_scale=30.0)
BATCHED_FP8 = Spec("batched_fp8", batch=8, seq=4896, heads=16, head_dim=64, rotary_dim=48,
                   grid=(16, 18, 17), in_dtype=BF16, out_kind=OUT_E4M3, scale_mode=SCALE_DYNAMIC,
                   outlier_frac=0.001, outlier_scale=30.0)
LATENT_65K = Spec("latent_65k", batch=1, seq=65280, heads=24, head_dim=128, rotary_dim=96,
                  grid=(32, 34, 60), in_dtype=BF16, outlier_frac=0.001, outlier_scale=50.0)
LATENT_65K_E4M3 = LATENT_65K.with_(name="latent_65k_e4m3", out_kind=OUT_E4M3,
                                   scale_mode=SCALE_DYNAMIC)
PREFIX_104K_STATIC = Spec("prefix_104k_static", batch=1, seq=104080, valid_len=104076, heads=40,
                          head_dim=128, rotary_dim=128, n_axes=1, in_dtype=BF16,
                          out_kind=OUT_E4M3, scale_mode=SCALE_STATIC, outlier_frac=0.0005,
                          outlier_scale=50.0)
PREFIX_104K_DYNAMIC = PREFIX_104K_STATIC.with_(name="prefix_104k_dynamic",
                                               scale_mode=SCALE_DYNAMIC)

WORKLOADS = {s.name: s for s in (TINY, DECODER_TILE, BATCHED_FP8, LATENT_65K, LATENT_65K_E4M3,
                                 PREFIX_104K_STATIC, PREFIX_104K_DYNAMIC)}
