"""Pins of the CPU oracle: checks against facts fixed by the pages, by the
number formats or by mathematics, never against the oracle's own formula.

Each ``pin_*`` function raises AssertionError when the oracle disagrees.
``tests/test_oracle_pins.py`` runs them one by one; ``tests/test_oracle_mutants.py``
runs the whole battery against deliberately broken copies of the oracle and
requires every copy to fail at least one pin.

Kinds of pin used here:
- library routines that compute the same special case (numpy's float16 and
  torch's bfloat16 / float8_e4m3fn conversions, libm's double sin/cos);
- closed forms and exact invariants (constant rows, power-of-two scaling,
  rotation by angle zero, axis separation, odd/even symmetry);
- brute force (integer rows whose sums are exact, amax by a second scan);
- the exact result within the error bound the rounding points allow (the
  whole path against a float64 evaluation of the plain mathematics);
- hand-worked values (``tests/golden/hand_worked.json``).
"""
from __future__ import annotations

import json
import math
import os
import re

import numpy as np

import oracle
from video_vae_decoder_qkv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers (format facts only)
# --------------------------------------------------------------------------

def _f16(codes):
    return np.asarray(codes, np.uint16).view(np.float16).astype(np.float64)


def _bf16(codes):
    return (np.asarray(codes, np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _widen(codes, dtype):
    return _f16(codes) if dtype == oracle.FP16 else _bf16(codes)


def _ulp16(v, dtype):
    """Spacing of the 16-bit format at |v| (the subnormal spacing below)."""
    mbits, emin = (10, -14) if dtype == oracle.FP16 else (7, -126)
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** emin)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - mbits)


QUICK = bool(os.environ.get("H3QK_PINS_QUICK"))


def _stratified_f32(seed=0, n_low=None):
    """fp32 bit patterns: every upper-16-bit pattern combined with low-16-bit
    patterns that sit on and around every rounding boundary of the 16-bit and
    8-bit formats (all-zero, half-way, one either side, all-ones) plus random
    ones; about 2^25 patterns."""
    n_low = n_low or (128 if QUICK else 512)
    rng = np.random.default_rng(seed)
    special = {0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0xFFFE}
    for b in range(16):
        h = 1 << b
        special |= {h, h - 1, h + 1, (h << 1) - 1 if b < 15 else 0xFFFF}
    lows = np.array(sorted(special | set(rng.integers(0, 1 << 16, n_low - len(special)).tolist())),
                    np.uint32)
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    return bits.view(np.float32)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def pin_f16_encoder():
    """binary32 -> binary16 RNE equals numpy's conversion on ~2^25 patterns
    around every rounding boundary (NaN: any quiet NaN with the sign)."""
    x = _stratified_f32()
    got = oracle.f32_to_f16(x)
    with np.errstate(over="ignore"):      # values past the binary16 range become infinities
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan]), "f16 encoder differs from numpy"
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)
    assert np.array_equal(got[nan] >> 15, (x[nan].view(np.uint32) >> 31).astype(np.uint16))


def pin_bf16_encoder():
    """binary32 -> bfloat16 RNE equals torch's conversion (finite values)."""
    import torch

    x = _stratified_f32(seed=1)
    got = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan]), "bf16 encoder differs from torch"
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


def pin_e4m3_encoder():
    """binary32 -> E4M3FN RNE equals torch's float8_e4m3fn conversion for
    every |x| < 448 of the stratified set; |x| >= 448 and infinities give
    0x7E / 0xFE (saturation, OCP 'satfinite'); NaN gives 0x7F / 0xFF."""
    import torch

    x = _stratified_f32(seed=2)
    got = oracle.f32_to_e4m3(x)
    fin = np.abs(x) < 448
    ref = torch.from_numpy(x[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[fin], ref), "e4m3 encoder differs from torch in range"
    big = (~fin) & ~np.isnan(x)
    sign = (x[big].view(np.uint32) >> 31).astype(np.uint8)
    assert np.array_equal(got[big], (0x7E | (sign << 7)).astype(np.uint8)), "e4m3 saturation"
    nan = np.isnan(x)
    assert np.all((got[nan] & 0x7F) == 0x7F)
    # every code's value round-trips (decode with torch, encode with the oracle)
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.f32_to_e4m3(vals[ok]), codes[ok])
    assert oracle.f32_to_e4m3(np.array([448.0 * 1.0001, 1e30, np.inf, -np.inf], np.float32)).tolist() \
        == [0x7E, 0x7E, 0x7E, 0xFE]


def pin_16b_decoders_roundtrip():
    """Every finite 16-bit code decodes (numpy / bit shift) and re-encodes to
    itself through the oracle's encoders."""
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = codes.view(np.float16).astype(np.float32)
    ok = np.isfinite(f)
    assert np.array_equal(oracle.f32_to_f16(f[ok]), codes[ok])
    b = (codes.astype(np.uint32) << 16).view(np.float32)
    ok = np.isfinite(b)
    assert np.array_equal(oracle.f32_to_bf16(b[ok]), codes[ok])


# --------------------------------------------------------------------------
# sine / cosine
# --------------------------------------------------------------------------

def _all_config_angles():
    out = []
    for spec in (W.TINY, W.DECODER_TILE, W.LATENT_65K, W.PREFIX_104K_STATIC):
        pb = _problem(spec)
        pos = W.positions(spec.with_(batch=1))
        pos = np.unique(pos, axis=0) if spec.n_axes == 3 else pos
        out.append(oracle.angles(pb, pos).reshape(-1))
    return np.unique(np.concatenate(out))


def pin_sincos_constants():
    """The reduction and series constants in the oracle source are the
    binary32 roundings of 2/pi, pi/2 split in three, and +-1/n!."""
    import mpmath

    mpmath.mp.prec = 200
    with open(oracle.source()) as f:
        src = f.read()

    def lit(name):
        m = re.search(r"H3O_%s\s*=\s*(-?0x[0-9a-fA-F.]+p[-+]?\d+)f;" % name, src)
        assert m, name
        return float.fromhex(m.group(1))

    def rn32(v):
        with mpmath.workprec(24):
            return float(+mpmath.mpf(v))

    assert lit("TWO_OVER_PI") == rn32(2 / mpmath.pi)
    p1 = rn32(mpmath.pi / 2)
    p2 = rn32(mpmath.pi / 2 - p1)
    p3 = rn32(mpmath.pi / 2 - p1 - p2)
    assert (lit("PIO2_1"), lit("PIO2_2"), lit("PIO2_3")) == (p1, p2, p3)
    for n in (3, 5, 7, 9, 11):
        assert lit("S%d" % n) == rn32((-1) ** ((n - 1) // 2) / mpmath.factorial(n)), n
    for n in (2, 4, 6, 8, 10, 12):
        assert lit("C%d" % n) == rn32((-1) ** (n // 2) / mpmath.factorial(n)), n


def pin_sincos_accuracy():
    """|sin - libm sin| and |cos - libm cos| <= 4 * 2^-24 over every angle the
    five workloads evaluate (libm in double precision); exact at 0; odd/even
    symmetry exact; s^2 + c^2 = 1 within 1e-6."""
    a = _all_config_angles()
    s, c = oracle.sincos(a)
    a64 = a.astype(np.float64)
    es = np.max(np.abs(s - np.sin(a64)))
    ec = np.max(np.abs(c - np.cos(a64)))
    assert es <= 4 * 2.0 ** -24 and ec <= 4 * 2.0 ** -24, (es, ec)
    s0, c0 = oracle.sincos(np.array([0.0], np.float32))
    assert s0[0] == 0.0 and not np.signbit(s0[0]) and c0[0] == 1.0
    sn, cn = oracle.sincos(-a)
    assert np.array_equal(sn, -s) and np.array_equal(cn, c)
    assert np.max(np.abs(s.astype(np.float64) ** 2 + c.astype(np.float64) ** 2 - 1)) <= 1e-6


def pin_sincos_addition():
    """Angle addition: c(a)c(b) - s(a)s(b) = c(a+b) and s(a)c(b) + c(a)s(b) =
    s(a+b) within 1e-6 for binary32 a, b with a+b exact."""
    rng = np.random.default_rng(5)
    a = np.float32(rng.integers(0, 4096, 20000)) * np.float32(2.0 ** -6)
    b = np.float32(rng.integers(0, 4096, 20000)) * np.float32(2.0 ** -6)
    sa, ca = [v.astype(np.float64) for v in oracle.sincos(a)]
    sb, cb = [v.astype(np.float64) for v in oracle.sincos(b)]
    sab, cab = [v.astype(np.float64) for v in oracle.sincos(a + b)]
    assert np.max(np.abs(ca * cb - sa * sb - cab)) <= 1e-6
    assert np.max(np.abs(sa * cb + ca * sb - sab)) <= 1e-6


def pin_inv_freq():
    """inv_freq[i] equals theta^(-2i/d) to within one binary32 ulp (mpmath)."""
    import mpmath

    mpmath.mp.prec = 100
    for theta, d in ((10000.0, 16), (10000.0, 32), (10000.0, 128), (500.0, 6)):
        got = oracle.inv_freq(theta, d).astype(np.float64)
        exact = np.array([float(mpmath.power(theta, mpmath.mpf(-2 * i) / d)) for i in range(d // 2)])
        assert got[0] == 1.0
        assert np.all(np.abs(got - exact) <= np.spacing(np.float32(exact)).astype(np.float64)), (theta, d)


# --------------------------------------------------------------------------
# per-head RMS normalisation
# --------------------------------------------------------------------------

def pin_sumsq_integers():
    """Integer rows whose partial sums stay below 2^24 are summed exactly in
    any order: the oracle's sum of squares equals the brute-force sum."""
    rng = np.random.default_rng(3)
    for D in (8, 16, 24, 64, 128, 136, 256):
        for _ in range(20):
            x = rng.integers(-180, 181, D).astype(np.float32)
            assert float(oracle.sumsq(x)) == float(np.sum(x.astype(np.int64) ** 2)), D


def pin_norm_unit_rms():
    """Before the weight, x * inv has mean square ms / (ms + eps) (relative
    1e-6), ms the exact mean square of x."""
    rng = np.random.default_rng(4)
    for D in (64, 128, 40):
        for scale in (1.0, 30.0, 1e-3):
            x = (rng.standard_normal(D) * scale).astype(np.float16).astype(np.float32)
            inv = float(oracle.rms_inv(x, 1e-6))
            ms = float(np.mean(x.astype(np.float64) ** 2))
            eps = float(np.float32(1e-6))
            got = float(np.mean((x.astype(np.float64) * inv) ** 2))
            assert abs(got - ms / (ms + eps)) <= 1e-6 * ms / (ms + eps) * 4, (D, scale)


def pin_norm_closed_forms():
    """Constant rows: n = c / sqrt(c^2 + eps) * w within one 16-bit ulp;
    power-of-two weights scale the rounded result exactly (weights applied
    channel by channel); with eps = 0, doubling x leaves n unchanged."""
    for dtype in (oracle.FP16, oracle.BF16):
        for c in (1.0, 0.5, 3.0, 0.0078125):
            for D in (64, 128):
                x = np.full(D, c, np.float32)
                n = _widen(oracle.norm_head(x, np.ones(D, np.float32), dtype), dtype)
                exact = c / math.sqrt(c * c + float(np.float32(1e-6)))
                assert np.all(np.abs(n - exact) <= _ulp16(exact, dtype)), (dtype, c, D)
        rng = np.random.default_rng(6)
        D = 128
        x = rng.standard_normal(D).astype(np.float32)
        x = _widen(oracle.f32_to_f16(x) if dtype == oracle.FP16 else oracle.f32_to_bf16(x), dtype).astype(np.float32)
        w = (2.0 ** (np.arange(D) % 3 - 1)).astype(np.float32)
        n1 = _widen(oracle.norm_head(x, np.ones(D, np.float32), dtype), dtype)
        nw = _widen(oracle.norm_head(x, w, dtype), dtype)
        assert np.array_equal(nw, n1 * w), "weights must scale channel by channel"
        a = _widen(oracle.norm_head(x, np.ones(D, np.float32), dtype, eps=0.0), dtype)
        b = _widen(oracle.norm_head(2 * x, np.ones(D, np.float32), dtype, eps=0.0), dtype)
        assert np.array_equal(a, b)


def pin_hand_worked():
    """Values worked by hand (tests/golden/hand_worked.json)."""
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        kind = case["kind"]
        if kind == "sumsq":
            got = float(oracle.sumsq(np.array(case["x"], np.float32)))
            assert got == case["expect"], (case["name"], got)
        elif kind == "rms_inv_bits":
            got = np.float32(oracle.rms_inv(np.array(case["x"], np.float32), case["eps"]))
            assert int(got.view(np.uint32)) == int(case["expect_bits"], 16), (case["name"], got)
        elif kind == "norm_f16":
            x = np.array(case["x"], np.float32)
            w = np.array(case["w"], np.float32)
            got = oracle.norm_head(x, w, oracle.FP16, case["eps"]).tolist()
            assert got == [int(h, 16) for h in case["expect_codes"]], (case["name"], [hex(g) for g in got])
        elif kind == "rotate_f16":
            got = oracle.rotate_pair(case["c"], case["s"], int(case["u"], 16), int(case["v"], 16))
            assert list(got) == [int(h, 16) for h in case["expect_codes"]], (case["name"], got)
        elif kind == "scaled_residual_f16":
            continue  # checked by pin_scaled_residual
        elif kind == "e4m3":
            got = oracle.f32_to_e4m3(np.array(case["x"], np.float32)).tolist()
            assert got == [int(h, 16) for h in case["expect_codes"]], (case["name"], got)
        else:
            raise AssertionError("unknown hand-worked kind " + kind)


# --------------------------------------------------------------------------
# rotary embedding
# --------------------------------------------------------------------------

def _problem(spec: W.Spec, **kw) -> oracle.Problem:
    d = dict(batch=spec.batch, seq=spec.seq, heads=spec.heads, head_dim=spec.head_dim,
             rotary_dim=spec.rotary_dim, n_axes=spec.n_axes, axis_dims=tuple(spec.axis_dims),
             in_dtype=spec.in_dtype, out_kind=spec.out_kind, scale_mode=spec.scale_mode,
             valid_len=spec.valid_len, row_stride=spec.row_stride, eps=spec.eps, theta=spec.theta)
    d.update(kw)
    return oracle.Problem(**d)


def _norm_only(inp: W.Inputs, pb: oracle.Problem, r: int):
    """The normalised (not rotated) 16-bit Q and K heads of row r."""
    D, HD = pb.head_dim, pb.hd
    row = inp.qkv[r]
    outs = []
    for part, w in ((0, inp.wq), (1, inp.wk)):
        heads = []
        for h in range(pb.heads):
            x = _widen(row[part * HD + h * D: part * HD + (h + 1) * D], pb.in_dtype).astype(np.float32)
            heads.append(oracle.norm_head(x, w, pb.in_dtype, pb.eps))
        outs.append(np.stack(heads))
    return outs


def pin_rope_identity_and_axes():
    """Position (0,0,0) leaves the normalised heads unchanged (exact); a
    position on one axis only changes that axis's channel segment; channels
    past rotary_dim are never rotated."""
    spec = W.TINY.with_(seq=4, grid=None, batch=1)
    for dtype in (oracle.FP16, oracle.BF16):
        inp = W.generate(spec.with_(in_dtype=dtype, seed=11))
        pb = _problem(inp.spec)
        pos = np.zeros((4, 3), np.int32)
        pos[1] = (5, 0, 0)
        pos[2] = (0, 7, 0)
        pos[3] = (0, 0, 9)
        yq, yk, _ = oracle.row16(pb, inp.qkv, inp.wq, inp.wk, pos, [0, 1, 2, 3])
        dims = pb.axis_dims
        seg = [(sum(dims[:a]), sum(dims[: a + 1])) for a in range(3)]
        for r in range(4):
            nq, nk = _norm_only(inp, pb, r)
            for y, n in ((yq[r], nq), (yk[r], nk)):
                assert np.array_equal(y[:, pb.rotary_dim:], n[:, pb.rotary_dim:])
                for a, (lo, hi) in enumerate(seg):
                    moved = r == a + 1
                    same = np.array_equal(y[:, lo:hi], n[:, lo:hi])
                    assert same != moved, (dtype, r, a)


def pin_rope_rotation_exact():
    """Each rotated pair is (u cos - v sin, u sin + v cos) of the normalised
    pair (u, v) = channels (2i, 2i+1), cos/sin of the angle pos[axis] *
    theta^(-2i/d_axis) evaluated in float64 from the binary32 angle, within
    the error the roundings allow (1.5 16-bit ulps of the pair plus 1 ulp of
    the result)."""
    for spec in (W.TINY, W.LATENT_65K.with_(seq=6, grid=(1, 2, 3)), W.PREFIX_104K_STATIC.with_(seq=5)):
        for dtype in (oracle.FP16, oracle.BF16):
            inp = W.generate(spec.with_(in_dtype=dtype, seed=12, valid_len=None))
            pb = _problem(inp.spec)
            pos = inp.pos.copy()
            pos[:] = np.random.default_rng(9).integers(0, 70000 if pb.n_axes == 1 else 64, pos.shape)
            rows = list(range(min(pb.rows, 6)))
            yq, yk, _ = oracle.row16(pb, inp.qkv, inp.wq, inp.wk, pos, rows)
            for r in rows:
                nq, nk = _norm_only(inp, pb, r)
                pair = 0
                ang = []
                for a, d in enumerate(pb.axis_dims):
                    for i in range(d // 2):
                        f = np.float32(float(pb.theta) ** (-(2.0 * i) / d))
                        ang.append(np.float32(np.float32(pos[r, a]) * f))
                        pair += 1
                ang = np.array(ang, np.float64)
                c, s = np.cos(ang), np.sin(ang)
                for y, n in ((yq[r], nq), (yk[r], nk)):
                    u = _widen(n[:, 0:pb.rotary_dim:2], dtype)
                    v = _widen(n[:, 1:pb.rotary_dim:2], dtype)
                    eu = u * c - v * s
                    ev = u * s + v * c
                    gu = _widen(y[:, 0:pb.rotary_dim:2], dtype)
                    gv = _widen(y[:, 1:pb.rotary_dim:2], dtype)
                    # u, v are exact 16-bit values: the only errors are two
                    # binary32 products, one binary32 sum (relative 2^-24 each),
                    # sin/cos (<= 4*2^-24 absolute) and the final 16-bit rounding
                    m = np.abs(u) + np.abs(v)
                    tol_u = 8 * 2.0 ** -24 * m + 0.5 * _ulp16(eu, dtype) * (1 + 2.0 ** -10)
                    tol_v = 8 * 2.0 ** -24 * m + 0.5 * _ulp16(ev, dtype) * (1 + 2.0 ** -10)
                    assert np.all(np.abs(gu - eu) <= tol_u), (spec.name, dtype, r)
                    assert np.all(np.abs(gv - ev) <= tol_v), (spec.name, dtype, r)


def pin_rotate_pair_exact():
    """One pair: the oracle's rotation equals the exactly rounded float64
    value (u c - v s, u s + v c) of its binary32 inputs, up to one 16-bit ulp
    (two binary32 roundings sit before the final 16-bit rounding)."""
    rng = np.random.default_rng(8)
    ang = rng.uniform(-7, 7, 4000).astype(np.float32)
    s, c = oracle.sincos(ang)
    u = rng.standard_normal(4000).astype(np.float16)
    v = rng.standard_normal(4000).astype(np.float16)
    for i in range(4000):
        gu, gv = oracle.rotate_pair(c[i], s[i], int(u[i:i + 1].view(np.uint16)[0]),
                                    int(v[i:i + 1].view(np.uint16)[0]))
        U, V, C, S = float(u[i]), float(v[i]), float(c[i]), float(s[i])
        eu, ev = U * C - V * S, U * S + V * C
        gu = float(np.uint16(gu).view(np.float16))
        gv = float(np.uint16(gv).view(np.float16))
        assert abs(gu - eu) <= _ulp16(eu, oracle.FP16) and abs(gv - ev) <= _ulp16(ev, oracle.FP16), i


# --------------------------------------------------------------------------
# the whole path
# --------------------------------------------------------------------------

def _exact_path(inp: W.Inputs, pb: oracle.Problem, r: int):
    """Float64 evaluation of the plain mathematics for row r: x / sqrt(mean
    x^2 + eps) * w, then the rotation by the binary32 angles; V copied."""
    D, HD, R = pb.head_dim, pb.hd, pb.rotary_dim
    row = inp.qkv[r]
    ang = []
    for a, d in enumerate(pb.axis_dims):
        for i in range(d // 2):
            f = np.float32(float(pb.theta) ** (-(2.0 * i) / d))
            ang.append(np.float32(np.float32(inp.pos[r, a]) * f))
    ang = np.array(ang, np.float64)
    c, s = np.cos(ang), np.sin(ang)
    eps = float(np.float32(pb.eps))
    res = []
    for part, w in ((0, inp.wq), (1, inp.wk)):
        x = _widen(row[part * HD: (part + 1) * HD], pb.in_dtype).reshape(pb.heads, D)
        n = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps) * w.astype(np.float64)
        y = n.copy()
        u, v = n[:, 0:R:2], n[:, 1:R:2]
        y[:, 0:R:2] = u * c - v * s
        y[:, 1:R:2] = u * s + v * c
        res.append((y, np.maximum(np.abs(u), np.abs(v))))
    vv = _widen(row[2 * HD: 3 * HD], pb.in_dtype).reshape(pb.heads, D)
    return res, vv


def pin_path_vs_float64():
    """Every Q and K value of the path lies within the error the stated
    rounding points allow of the float64 mathematics (two 16-bit roundings:
    |err| <= 1.5 ulp16(pair) + ulp16(value) + 2^-20 |value|), V is bit-exact;
    on the tiny workload and on 16-bit/bfloat16 variants of the others."""
    cases = [W.TINY, W.DECODER_TILE.with_(seq=40, grid=(2, 4, 5)),
             W.LATENT_65K.with_(seq=12, grid=(1, 3, 4), in_dtype=oracle.FP16),
             W.PREFIX_104K_STATIC.with_(seq=9, out_kind=0, scale_mode=0, valid_len=None)]
    for spec in cases:
        inp = W.generate(spec)
        pb = _problem(inp.spec)
        rows = list(range(pb.rows))
        yq, yk, yv = oracle.row16(pb, inp.qkv, inp.wq, inp.wk, inp.pos, rows)
        for r in rows:
            ((eq, mq), (ek, mk)), ev = _exact_path(inp, pb, r)
            for g, e, m in ((yq[r], eq, mq), (yk[r], ek, mk)):
                gv = _widen(g, pb.in_dtype)
                tol = _ulp16(e, pb.in_dtype) + 2.0 ** -20 * np.abs(e)
                R = pb.rotary_dim
                tol[:, :R] += np.repeat(1.5 * _ulp16(m, pb.in_dtype), 2, axis=1)
                assert np.all(np.abs(gv - e) <= tol), (spec.name, r, np.max(np.abs(gv - e) - tol))
            assert np.array_equal(_widen(yv[r], pb.in_dtype), ev)


def pin_layout_bruteforce():
    """Head-major placement: with every input element a distinct code, the
    V output at [b, h, s, d] is the input at row b*S+s, column 2HD + h*D + d,
    and the Q/K output at [b, h, s] is head h of the per-row result of row
    b*S+s (brute force over every element)."""
    spec = W.TINY.with_(batch=2, seq=24, grid=(2, 3, 4), dist="unique")
    inp = W.generate(spec)
    pb = _problem(inp.spec)
    q, k, v, _ = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
    H, D, S, HD = pb.heads, pb.head_dim, pb.seq, pb.hd
    yq, yk, _ = oracle.row16(pb, inp.qkv, inp.wq, inp.wk, inp.pos, range(pb.rows))
    for b in range(pb.batch):
        for h in range(H):
            for s in range(S):
                r = b * S + s
                for d in range(D):
                    assert v[b, h, s, d] == inp.qkv[r, 2 * HD + h * D + d]
                assert np.array_equal(q[b, h, s], yq[r, h]) and np.array_equal(k[b, h, s], yk[r, h])


def pin_amax_scales_cast():
    """amax equals a brute-force max |y| over the valid rows of the 16-bit
    path's output; the dynamic descale is amax/448 and the amax element
    encodes to 0x7E/0xFE; every code equals torch's e4m3 conversion of
    y * (448/amax) when in range and saturates otherwise; a static table of
    small descales saturates a counted fraction."""
    import torch

    base = W.BATCHED_FP8.with_(batch=2, seq=48, grid=(2, 4, 6), valid_len=45)
    inp = W.generate(base)
    pb16 = _problem(base, out_kind=0, scale_mode=0)
    q16, k16, v16, _ = oracle.prepare(pb16, inp.qkv, inp.wq, inp.wk, inp.pos)
    vl = base.valid_len
    brute = np.array([np.max(np.abs(_widen(t[:, :, :vl], base.in_dtype))) for t in (q16, k16, v16)])
    pbd = _problem(base)
    am = oracle.amax(pbd, inp.qkv, inp.wq, inp.wk, inp.pos)
    assert np.array_equal(am.astype(np.float64), brute), (am, brute)
    q8, k8, v8, sc = oracle.prepare(pbd, inp.qkv, inp.wq, inp.wk, inp.pos)
    for t, (c8, c16) in enumerate(((q8, q16), (k8, k16), (v8, v16))):
        assert sc[t] == np.float32(am[t]) / np.float32(448.0)
        y = _widen(c16[:, :, :vl], base.in_dtype).astype(np.float32)
        z = (y * (np.float32(448.0) / np.float32(am[t]))).astype(np.float32)
        codes = c8[:, :, :vl]
        inr = np.abs(z) < 448
        ref = torch.from_numpy(z[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes[inr], ref)
        assert np.all((codes[~inr] & 0x7F) == 0x7E)
        arg = np.argmax(np.abs(y))
        assert (codes.reshape(-1)[arg] & 0x7F) == 0x7E
        assert np.all(c8[:, :, vl:] == 0), "padded rows must stay untouched"
    pbs = _problem(base, scale_mode=oracle.SCALE_STATIC, static_scales=(0.01, 0.02, 0.5))
    q8, k8, v8, sc = oracle.prepare(pbs, inp.qkv, inp.wq, inp.wk, inp.pos)
    assert sc.tolist() == [np.float32(0.01), np.float32(0.02), np.float32(0.5)]
    sat = [np.mean((t[:, :, :vl] & 0x7F) == 0x7E) for t in (q8, k8, v8)]
    assert sat[0] > 0 and sat[1] > 0 and sat[2] == 0, sat


def pin_valid_prefix():
    """Rows past valid_len keep the output buffer's bytes and are left out of
    the amax: filling them with huge values changes nothing."""
    base = W.DECODER_TILE.with_(batch=2, seq=30, grid=(2, 3, 5), valid_len=27, in_dtype=oracle.BF16)
    inp = W.generate(base)
    pb = _problem(base, out_kind=oracle.OUT_E4M3, scale_mode=oracle.SCALE_DYNAMIC)
    a0 = oracle.amax(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
    huge = inp.qkv.copy()
    for b in range(base.batch):
        huge[b * base.seq + base.valid_len:(b + 1) * base.seq] = 0x7F00   # bf16 ~1.7e38
    a1 = oracle.amax(pb, huge, inp.wq, inp.wk, inp.pos)
    assert np.array_equal(a0, a1)
    shape = (base.batch, base.heads, base.seq, base.head_dim)
    canary = tuple(np.full(shape, 0xA5, np.uint8) for _ in range(3))
    q, k, v, _ = oracle.prepare(pb, huge, inp.wq, inp.wk, inp.pos, out=canary)
    for t in (q, k, v):
        assert np.all(t[:, :, base.valid_len:] == 0xA5)
        assert not np.all(t[:, :, : base.valid_len] == 0xA5)
    pb16 = _problem(base)
    c16 = tuple(np.full(shape, 0x5A5A, np.uint16) for _ in range(3))
    q, k, v, _ = oracle.prepare(pb16, huge, inp.wq, inp.wk, inp.pos, out=c16)
    for t in (q, k, v):
        assert np.all(t[:, :, base.valid_len:] == 0x5A5A)


def pin_batch_items_independent():
    """In 16-bit mode each item of a batch equals a batch-1 run on its rows
    (positions are tile-local, nothing couples the items)."""
    base = W.DECODER_TILE.with_(batch=3, seq=20, grid=(1, 4, 5))
    inp = W.generate(base)
    pb = _problem(base)
    q, k, v, _ = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
    pb1 = _problem(base, batch=1)
    for b in range(3):
        sl = slice(b * 20, (b + 1) * 20)
        q1, k1, v1, _ = oracle.prepare(pb1, inp.qkv[sl], inp.wq, inp.wk, inp.pos[sl])
        assert np.array_equal(q[b], q1[0]) and np.array_equal(k[b], k1[0]) and np.array_equal(v[b], v1[0])


def pin_threads_equal_serial():
    """Row ranges on several threads give the same bytes as one thread."""
    base = W.BATCHED_FP8.with_(batch=2, seq=48, grid=(2, 4, 6))
    inp = W.generate(base)
    for pb in (_problem(base), _problem(base, out_kind=0, scale_mode=0)):
        a = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos, threads=1)
        b = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos, threads=3)
        for x, y in zip(a[:3], b[:3]):
            assert np.array_equal(x, y)
        if a[3] is not None:
            assert np.array_equal(a[3], b[3])


def pin_golden_digest():
    """The oracle's outputs on the tiny workloads still hash to the digests
    written by tests/golden/make_golden.py (a regression pin: any change to
    the oracle's arithmetic must rewrite them in a commit that says why)."""
    import hashlib

    with open(os.path.join(GOLDEN, "oracle_digests.json")) as f:
        ref = json.load(f)
    for name, want in ref["digests"].items():
        spec, pb_kw = GOLDEN_CASES[name]
        inp = W.generate(spec)
        pb = _problem(spec, **pb_kw)
        q, k, v, sc = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
        h = hashlib.sha256()
        for t in (q, k, v):
            h.update(np.ascontiguousarray(t).tobytes())
        if sc is not None:
            h.update(np.asarray(sc, np.float32).tobytes())
        assert h.hexdigest() == want, name


GOLDEN_CASES = {
    "tiny_fp16": (W.TINY, {}),
    "tiny_bf16": (W.TINY.with_(in_dtype=W.BF16), {}),
    "tiny_bf16_e4m3_dynamic": (W.TINY.with_(in_dtype=W.BF16, out_kind=W.OUT_E4M3,
                                            scale_mode=W.SCALE_DYNAMIC), {}),
    "tiny_fp16_e4m3_static_prefix": (W.TINY.with_(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC,
                                                  valid_len=45, n_axes=1, rotary_dim=64, grid=None),
                                     {"static_scales": (0.01, 0.02, 0.05)}),
}


PINS = [pin_f16_encoder, pin_bf16_encoder, pin_e4m3_encoder, pin_16b_decoders_roundtrip,
        pin_sincos_constants, pin_sincos_accuracy, pin_sincos_addition, pin_inv_freq,
        pin_sumsq_integers, pin_norm_unit_rms, pin_norm_closed_forms, pin_hand_worked,
        pin_rope_identity_and_axes, pin_rope_rotation_exact, pin_rotate_pair_exact,
        pin_path_vs_float64, pin_layout_bruteforce, pin_amax_scales_cast, pin_valid_prefix,
        pin_batch_items_independent, pin_threads_equal_serial, pin_golden_digest]


def run_all() -> list[str]:
    """Run every pin; return the names of those that failed."""
    failed = []
    for p in PINS:
        try:
            p()
        except Exception as e:  # noqa: BLE001 - a mutant may fail in any way
            failed.append(f"{p.__name__}: {type(e).__name__}: {str(e)[:120]}")
    return failed


# --------------------------------------------------------------------------
# options: token-major output, per-item valid lengths, saturation counts,
# the single-tensor variant
# --------------------------------------------------------------------------

def pin_token_major_layout():
    """Token-major output holds, at [b, s, h, :], exactly what head-major
    output holds at [b, h, s, :] (brute force over every element)."""
    spec = W.TINY.with_(batch=2, seq=24, grid=(2, 3, 4), dist="unique")
    inp = W.generate(spec)
    hm = oracle.prepare(_problem(spec), inp.qkv, inp.wq, inp.wk, inp.pos)
    tm = oracle.prepare(_problem(spec, out_layout=1), inp.qkv, inp.wq, inp.wk, inp.pos)
    for a, b in zip(hm[:3], tm[:3]):
        assert b.shape == (2, 24, 4, 64)
        for bb in range(2):
            for s in range(24):
                for h in range(4):
                    assert np.array_equal(b[bb, s, h], a[bb, h, s])


def pin_per_item_valid_lengths():
    """Per-item lengths (0, S, a middle value, one out of range) keep each
    item's own prefix: canaries past it survive, rows before it equal an
    all-valid run, and huge values past it leave the amax unchanged."""
    spec = W.BATCHED_FP8.with_(batch=4, seq=20, grid=(1, 4, 5), in_dtype=oracle.BF16)
    inp = W.generate(spec)
    lens = (0, 20, 7, 99)
    eff = (0, 20, 7, 20)
    for kind in (0, 1):
        pbv = _problem(spec, out_kind=kind, scale_mode=kind, valid_lens=lens)
        pba = _problem(spec, out_kind=0, scale_mode=0)
        odt = np.uint8 if kind else np.uint16
        fill = 0xA5 if kind else 0x5A5A
        shape = (4, spec.heads, 20, spec.head_dim)
        out = tuple(np.full(shape, fill, odt) for _ in range(3))
        got = oracle.prepare(pbv, inp.qkv, inp.wq, inp.wk, inp.pos, out=out)
        full = oracle.prepare(pba, inp.qkv, inp.wq, inp.wk, inp.pos)
        for t in range(3):
            for b in range(4):
                assert np.all(got[t][b, :, eff[b]:] == fill)
                if kind == 0:
                    assert np.array_equal(got[t][b, :, :eff[b]], full[t][b, :, :eff[b]])
    pbd = _problem(spec, out_kind=1, scale_mode=1, valid_lens=lens)
    huge = inp.qkv.copy()
    for b in range(4):
        huge[b * 20 + eff[b]:(b + 1) * 20] = 0x7F00
    assert np.array_equal(oracle.amax(pbd, inp.qkv, inp.wq, inp.wk, inp.pos),
                          oracle.amax(pbd, huge, inp.wq, inp.wk, inp.pos))


def pin_saturation_counts():
    """Counts equal a brute-force count (numpy) of |y * inv| > 448 over the
    16-bit outputs; a tiny descale saturates every non-zero value, a huge one
    none, and dynamic scales clip at most the amax element."""
    spec = W.BATCHED_FP8.with_(batch=2, seq=40, grid=(1, 5, 8), valid_len=37)
    inp = W.generate(spec)
    pb16 = _problem(spec, out_kind=0, scale_mode=0)
    y = oracle.prepare(pb16, inp.qkv, inp.wq, inp.wk, inp.pos)[:3]
    vals = [_widen(t[:, :, :37], spec.in_dtype).astype(np.float32) for t in y]
    pb = _problem(spec)
    for inv in ([1.0, 1.0, 1.0], [100.0, 30.0, 200.0], [1e30, 1e30, 1e30], [1e-30, 1e-30, 1e-30]):
        got = oracle.sat_counts(pb, inp.qkv, inp.wq, inp.wk, inp.pos, np.array(inv, np.float32))
        want = [int(np.sum(np.abs((v * np.float32(f)).astype(np.float32)) > 448)) for v, f in zip(vals, inv)]
        assert got.tolist() == want, (inv, got, want)
    nz = [int(np.sum(v != 0)) for v in vals]
    assert oracle.sat_counts(pb, inp.qkv, inp.wq, inp.wk, inp.pos, np.full(3, 1e30, np.float32)).tolist() == nz
    # exactly +-448 is the largest code, not clipped; 450 is clipped (V passes
    # its input through, so these values reach the cast unchanged)
    edge = inp.qkv.copy()
    v0 = 2 * spec.hd
    edge[0, v0:v0 + 4] = np.array([448.0, -448.0, 450.0, 446.0], np.float32).view(np.uint32) >> 16
    edge[1, v0:v0 + 4] = np.array([448.0, 448.0, -450.0, 0.0], np.float32).view(np.uint32) >> 16
    one = oracle.sat_counts(pb, edge, inp.wq, inp.wk, inp.pos, np.ones(3, np.float32))
    vv = _widen(oracle.prepare(pb16, edge, inp.wq, inp.wk, inp.pos)[2][:, :, :37], spec.in_dtype)
    assert int(one[2]) == int(np.sum(np.abs(vv) > 448)) == 2
    am = oracle.amax(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
    _, inv = oracle.scales(pb, am)
    assert all(c <= 1 for c in oracle.sat_counts(pb, inp.qkv, inp.wq, inp.wk, inp.pos, inv).tolist())


def pin_single_tensor_matches_packed():
    """The single-tensor path on the Q (K, V) slice of packed rows gives the
    packed path's Q (K, V) output, token-major; its e4m3 amax equals a
    brute-force max over its 16-bit output."""
    spec = W.DECODER_TILE.with_(batch=2, seq=30, grid=(1, 5, 6), valid_len=27, in_dtype=oracle.BF16)
    inp = W.generate(spec)
    HD = spec.hd
    pbp = _problem(spec, out_layout=1)
    packed = oracle.prepare(pbp, inp.qkv, inp.wq, inp.wk, inp.pos)
    for kind, w in ((0, inp.wq), (1, inp.wk), (2, None)):
        x = np.ascontiguousarray(inp.qkv[:, kind * HD:(kind + 1) * HD])
        pbt = oracle.Problem(batch=2, seq=30, heads=spec.heads, head_dim=spec.head_dim,
                             rotary_dim=spec.rotary_dim, in_dtype=spec.in_dtype, valid_len=27, tensor=True)
        out, _ = oracle.tensor_prepare(pbt, kind, x, w, inp.pos)
        assert np.array_equal(out[:, :27], packed[kind][:, :27])
        pbd = oracle.Problem(batch=2, seq=30, heads=spec.heads, head_dim=spec.head_dim,
                             rotary_dim=spec.rotary_dim, in_dtype=spec.in_dtype, valid_len=27, tensor=True,
                             out_kind=1, scale_mode=1)
        codes, scale = oracle.tensor_prepare(pbd, kind, x, w, inp.pos)
        brute = float(np.max(np.abs(_widen(out[:, :27], spec.in_dtype))))
        assert scale == np.float32(np.float32(brute) / np.float32(448.0))


PINS += [pin_token_major_layout, pin_per_item_valid_lengths, pin_saturation_counts,
         pin_single_tensor_matches_packed]


# --------------------------------------------------------------------------
# adjacent VAE-block operations: e^x, SiLU, SwiGLU, scaled residual
# --------------------------------------------------------------------------

def pin_exp():
    """e^x: the constants are the binary32 roundings of log2(e), ln2 and its
    tail, 1/n!; |e^x - libm| <= 2^-23 relative over [-17.5, 88.72] (2 M
    points); exact at 0; e^x e^-x = 1 within 2^-22; NaN, overflow and the
    cut-off below 2^-126."""
    import mpmath

    mpmath.mp.prec = 200
    with open(oracle.source()) as f:
        src = f.read()

    def lit(name):
        m = re.search(r"H3O_%s\s*=\s*(-?0x[0-9a-fA-F.]+p[-+]?\d+)f;" % name, src)
        assert m, name
        return float.fromhex(m.group(1))

    def rn32(v):
        with mpmath.workprec(24):
            return float(+mpmath.mpf(v))

    assert lit("LOG2E") == rn32(1 / mpmath.log(2))
    hi = rn32(mpmath.log(2))
    assert (lit("LN2_HI"), lit("LN2_LO")) == (hi, rn32(mpmath.log(2) - hi))
    for n in range(2, 9):
        assert lit("E%d" % n) == rn32(1 / mpmath.factorial(n)), n
    x = np.linspace(-17.5, 88.72, 2_000_001).astype(np.float32)
    y = oracle.exp(x).astype(np.float64)
    t = np.exp(x.astype(np.float64))
    assert np.max(np.abs(y - t) / t) <= 2.0 ** -23
    assert oracle.lib().h3o_exp(0.0) == 1.0
    z = np.float32(np.linspace(-17, 17, 10001))
    assert np.max(np.abs(oracle.exp(z).astype(np.float64) * oracle.exp(-z) - 1)) <= 2.0 ** -22
    assert np.isnan(oracle.lib().h3o_exp(float("nan")))
    assert oracle.lib().h3o_exp(100.0) == float("inf") and oracle.lib().h3o_exp(-110.0) == 0.0


def pin_silu():
    """SiLU: 0 at 0; exactly g once 1 + e^-g rounds to 1 (g >= 17.4);
    within 4 binary32 ulps of g / (1 + exp(-g)) in float64 elsewhere; the odd
    part silu(g) - silu(-g) = g within the same bound."""
    L = oracle.lib()
    assert L.h3o_silu(0.0) == 0.0
    for g in (17.5, 20.0, 1000.0, 65504.0):
        assert L.h3o_silu(g) == np.float32(g)
    g = np.float32(np.linspace(-30, 30, 20001))
    got = np.array([L.h3o_silu(float(v)) for v in g], np.float64)
    ref = g.astype(np.float64) / (1 + np.exp(-g.astype(np.float64)))
    tol = 4 * np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) + 1e-45
    assert np.all(np.abs(got - ref) <= tol)
    neg = np.array([L.h3o_silu(float(-v)) for v in g], np.float64)
    assert np.all(np.abs((got - neg) - g) <= 8 * np.spacing(np.abs(g)).astype(np.float64) + 1e-40)


def pin_swiglu():
    """SwiGLU rows: gate from the first half, up from the second; every value
    within one 16-bit ulp (plus the binary32 errors) of silu(gate) * up in
    float64; row stride larger than 2f respected."""
    rng = np.random.default_rng(31)
    for dtype, to16, wid in ((oracle.FP16, oracle.f32_to_f16, _f16), (oracle.BF16, oracle.f32_to_bf16, _bf16)):
        rows, f, stride = 7, 24, 56
        x = to16(rng.standard_normal(rows * stride).astype(np.float32) * 3).reshape(rows, stride)
        out = oracle.silu_and_mul(x, f, dtype)
        g = wid(x[:, :f])
        u = wid(x[:, f:2 * f])
        ref = g / (1 + np.exp(-g)) * u
        got = wid(out)
        tol = _ulp16(ref, dtype) + 8 * 2.0 ** -24 * np.abs(ref)
        assert np.all(np.abs(got - ref) <= tol), dtype


def pin_scaled_residual():
    """Power-of-two scales make the product exact, so out equals the
    correctly rounded float64 sum; per-channel scales pick their own channel;
    a scalar scale broadcasts; the hand-worked case shows the product's own
    rounding (tests/golden/hand_worked.json)."""
    rng = np.random.default_rng(32)
    rows, C = 5, 16
    res = rng.standard_normal((rows, C)).astype(np.float32)
    br = oracle.f32_to_f16(rng.standard_normal(rows * C).astype(np.float32)).reshape(rows, C)
    s = (2.0 ** rng.integers(-3, 4, C)).astype(np.float32)
    out = oracle.scaled_residual(res, br, s, oracle.FP16)
    exact = (res.astype(np.float64) + _f16(br) * s.astype(np.float64)).astype(np.float32)
    assert np.array_equal(out, exact)
    one = oracle.scaled_residual(res, br, np.array([0.5], np.float32), oracle.FP16)
    assert np.array_equal(one, (res.astype(np.float64) + _f16(br) * 0.5).astype(np.float32))
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = [c for c in json.load(f)["cases"] if c["kind"] == "scaled_residual_f16"]
    assert cases
    for c in cases:
        o = oracle.scaled_residual(np.array([[c["residual"]] * 8], np.float32),
                                   np.array([[int(c["branch"], 16)] * 8], np.uint16),
                                   np.array([c["scale"]], np.float32), oracle.FP16)
        assert float(o[0, 0]) == c["expect"], (c["name"], float(o[0, 0]))


PINS += [pin_exp, pin_silu, pin_swiglu, pin_scaled_residual]


# --------------------------------------------------------------------------
# sage-attention outputs: F32 Q, F32 K * kv_scale, F16 V * kv_scale
# --------------------------------------------------------------------------

def _sage_spec(dtype, **kw):
    d = dict(name="sage", batch=2, seq=30, grid=(2, 3, 5), valid_len=None, in_dtype=dtype)
    d.update(kw)
    return W.LATENT_65K.with_(**d)


def _head_index(pb, r, h):
    b, s = divmod(r, pb.seq)
    return (b, s, h) if pb.out_layout == 1 else (b, h, s)


def pin_sage_vs_float64():
    """Q and K of the sage outputs lie within binary32 error of the float64
    mathematics (x / sqrt(mean x^2 + eps) * w, rotated by the binary32
    angles; K times kv_scale): |err| <= 2^-17 (|u| + |v|) on rotated pairs
    and 2^-17 |n| elsewhere.  A 16-bit rounding anywhere in the chain
    (2^-11 or 2^-8 relative) or a misplaced kv_scale breaks it.  Checked at
    every (b, h, s) of both layouts, so the placement is pinned too."""
    for dtype in (oracle.FP16, oracle.BF16):
        for layout in (0, 1):
            spec = _sage_spec(dtype)
            inp = W.generate(spec)
            pb = _problem(spec, out_layout=layout)
            kvs = 0.3
            q, k, v = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, inp.pos, kv_scale=kvs)
            R = pb.rotary_dim
            for r in range(pb.rows):
                ((eq, _), (ek, _)), _ = _exact_path(inp, pb, r)
                # pre-rotation magnitudes from the float64 norm
                for got_t, e, scale in ((q, eq, 1.0), (k, ek, kvs)):
                    for h in range(pb.heads):
                        g = got_t[_head_index(pb, r, h)].astype(np.float64)
                        ee = e[h] * scale
                        mag = np.abs(ee).copy()
                        pair = np.abs(ee[0:R:2]) + np.abs(ee[1:R:2])
                        mag[0:R:2] = pair
                        mag[1:R:2] = pair
                        tol = 2.0 ** -17 * mag + 1e-30
                        assert np.all(np.abs(g - ee) <= tol), (dtype, layout, r, h, np.max(np.abs(g - ee) / tol))


def pin_sage_v_matches_numpy():
    """V codes equal numpy's binary16 conversion of float32(v) *
    float32(kv_scale) for both input types, including products that
    overflow binary16 (to infinity) and land in its subnormal range."""
    for dtype in (oracle.FP16, oracle.BF16):
        spec = _sage_spec(dtype, batch=1, seq=12, grid=(1, 3, 4))
        inp = W.generate(spec)
        pb = _problem(spec)
        HD = pb.hd
        for kvs in (1.0, 0.3, 3.0e4, 1.0e-6):
            _, _, v = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, inp.pos, kv_scale=kvs)
            for r in range(pb.rows):
                x = _widen(inp.qkv[r, 2 * HD:3 * HD], dtype).astype(np.float32)
                with np.errstate(over="ignore"):  # products past the binary16 range become infinities
                    want = (x * np.float32(kvs)).astype(np.float16).view(np.uint16).reshape(pb.heads, -1)
                for h in range(pb.heads):
                    assert np.array_equal(v[_head_index(pb, r, h)], want[h]), (dtype, kvs, r, h)


def pin_sage_agrees_with_16bit_path():
    """Where the rotation is the identity (position (0, 0, 0): cos 1, sin 0)
    or absent (rotary_dim 0), the 16-bit rounding of the sage Q and K (with
    kv_scale 1) is the 16-bit path's output, code for code: the two differ
    only in where the 16-bit rounding sits."""
    for dtype in (oracle.FP16, oracle.BF16):
        for rd in (48, 0):
            spec = _sage_spec(dtype, rotary_dim=rd, axis_dims=(16, 16, 16) if rd else (0, 0, 0))
            inp = W.generate(spec)
            pos = np.zeros_like(inp.pos) if rd else inp.pos
            pb = _problem(spec)
            q, k, _ = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, pos, kv_scale=1.0)
            q16, k16, _, _ = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, pos)
            conv = oracle.f32_to_f16 if dtype == oracle.FP16 else oracle.f32_to_bf16
            for a, b in ((q, q16), (k, k16)):
                assert np.array_equal(conv(a.reshape(-1)).reshape(a.shape), b), (dtype, rd)


def pin_sage_kv_scale_and_prefix():
    """A power-of-two kv_scale scales K exactly (K(2^-3) = K(1) / 8) and
    leaves Q alone; rows past each item's valid length keep the canary."""
    spec = _sage_spec(oracle.BF16)
    inp = W.generate(spec)
    pb = _problem(spec)
    q1, k1, _ = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, inp.pos, kv_scale=1.0)
    q8, k8, _ = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, inp.pos, kv_scale=0.125)
    assert np.array_equal(q1.view(np.uint32), q8.view(np.uint32))
    assert np.array_equal(k8, k1 / np.float32(8))
    pbv = _problem(spec, valid_len=17)
    shape = q1.shape
    canary = (np.full(shape, np.float32(-7.25)), np.full(shape, np.float32(-7.25)),
              np.full(shape, 0x5A5A, np.uint16))
    qv, kv, vv = oracle.sage(pbv, inp.qkv, inp.wq, inp.wk, inp.pos, kv_scale=1.0, out=canary)
    _, _, v1 = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, inp.pos, kv_scale=1.0)
    for got, full in ((qv, q1), (kv, k1), (vv, v1)):
        assert np.array_equal(got[:, :, :17], full[:, :, :17])
        assert np.all(got[:, :, 17:] == (0x5A5A if got.dtype == np.uint16 else np.float32(-7.25)))


PINS += [pin_sage_vs_float64, pin_sage_v_matches_numpy, pin_sage_agrees_with_16bit_path,
         pin_sage_kv_scale_and_prefix]


# --------------------------------------------------------------------------
# degenerate scales and non-finite values (readings of the cast and of
# IEEE propagation; the pages are silent on both)
# --------------------------------------------------------------------------

_FLT_MIN = np.float32(np.finfo(np.float32).tiny)
_FLT_MAX = np.float32(np.finfo(np.float32).max)


def pin_scales_degenerate():
    """A descale needs a finite, normal, positive binary32.  Zero (either
    sign), the largest and smallest subnormals, infinities, NaN and negative
    values give scale = factor = 1 in both modes.  Normal values, the two ends
    of the normal range included, give amax/448 and 448/amax (dynamic) or the
    entry and its reciprocal (static).  Each is one IEEE binary32 division,
    which numpy's float32 arithmetic performs."""
    bad = [0.0, -0.0, np.nextafter(_FLT_MIN, np.float32(0)), np.float32(1e-40), np.float32(2.0 ** -149),
           np.inf, -np.inf, np.nan, -1.0, -_FLT_MIN]
    good = [_FLT_MIN, np.nextafter(_FLT_MIN, np.float32(1)), np.float32(1e-20), np.float32(0.37),
            np.float32(448.0), np.float32(3.5e37), _FLT_MAX]
    base = W.TINY.with_(out_kind=W.OUT_E4M3)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        for mode in (oracle.SCALE_DYNAMIC, oracle.SCALE_STATIC):
            for vals in ([bad[i % len(bad)] for i in range(k, k + 3)] for k in range(len(bad))):
                a = np.array(vals, np.float32)
                pb = _problem(base, scale_mode=mode, static_scales=tuple(float(x) for x in a))
                s, f = oracle.scales(pb, a)
                assert s.tolist() == [1.0] * 3 and f.tolist() == [1.0] * 3, (mode, vals, s, f)
            for vals in ([good[i % len(good)] for i in range(k, k + 3)] for k in range(len(good))):
                a = np.array(vals, np.float32)
                pb = _problem(base, scale_mode=mode, static_scales=tuple(float(x) for x in a))
                s, f = oracle.scales(pb, a)
                if mode == oracle.SCALE_DYNAMIC:
                    ws, wf = a / np.float32(448.0), np.float32(448.0) / a
                else:
                    ws, wf = a, np.float32(1.0) / a
                assert np.array_equal(s.view(np.uint32), ws.astype(np.float32).view(np.uint32)), (vals, s, ws)
                assert np.array_equal(f.view(np.uint32), wf.astype(np.float32).view(np.uint32)), (vals, f, wf)
            # a mixed table: only the degenerate entries fall back
            a = np.array([0.0, np.float32(0.25), np.nan], np.float32)
            pb = _problem(base, scale_mode=mode, static_scales=tuple(float(x) for x in a))
            s, f = oracle.scales(pb, a)
            mid = (np.float32(0.25) / np.float32(448.0), np.float32(448.0) / np.float32(0.25)) \
                if mode == oracle.SCALE_DYNAMIC else (np.float32(0.25), np.float32(4.0))
            assert s.tolist() == [1.0, float(mid[0]), 1.0] and f.tolist() == [1.0, float(mid[1]), 1.0], (s, f)


def _bf16_code(x: float) -> int:
    """bfloat16 code of a value that bfloat16 holds exactly (or inf / NaN)."""
    return int(np.array([x], np.float32).view(np.uint32)[0] >> 16)


def pin_nonfinite_values():
    """NaN and infinity follow IEEE arithmetic through the path, and the amax
    leaves NaN out.
    - A NaN input channel makes the head's sum of squares NaN, so every
      channel of that Q head comes out NaN, and the other heads are unchanged.
    - An infinite K channel makes the sum infinite and 1/sqrt of it zero.
      That channel becomes inf * 0 = NaN, and so does its rotation partner.
      Every other channel of the head becomes a signed zero.
    - V passes NaN and infinity through unchanged.
    - The amax is the maximum |y| over the values that are not NaN: a
      numpy nanmax over the 16-bit output, never NaN itself.  An infinite V
      value gives an infinite amax, hence the fallback scale 1 and factor 1.
      The infinity then saturates to the largest code (0x7E, sign kept), NaN
      gives a NaN code, and the finite values equal torch's e4m3 conversion.
    - The single-tensor path's amax skips NaN in the same way."""
    import torch

    spec = W.TINY.with_(in_dtype=W.BF16, batch=1, seq=12, grid=(1, 3, 4), valid_len=12)
    inp = W.generate(spec)
    H, D, HD = spec.heads, spec.head_dim, spec.hd
    x = inp.qkv.copy()
    nan16, inf16 = 0x7FC0, _bf16_code(np.inf)
    x[2, 1 * D + 5] = nan16                 # Q row 2, head 1, channel 5
    x[4, HD + 0 * D + 7] = inf16            # K row 4, head 0, channel 7 (pair 3, rotated)
    x[3, 2 * HD + 2 * D + 9] = nan16        # V row 3, head 2, channel 9
    x[11, 3 * HD - 1] = nan16               # and the very last V value scanned
    pb16 = _problem(spec, out_kind=0, scale_mode=0)
    q, k, v, _ = oracle.prepare(pb16, x, inp.wq, inp.wk, inp.pos)
    q0, k0, v0, _ = oracle.prepare(pb16, inp.qkv, inp.wq, inp.wk, inp.pos)
    qf, kf, vf = (_widen(t, spec.in_dtype) for t in (q, k, v))
    assert np.all(np.isnan(qf[0, 1, 2])), "a NaN channel must make its whole Q head NaN"
    others = [h for h in range(H) if h != 1]
    assert np.array_equal(q[0, others, 2], q0[0, others, 2]), "other heads of the row must not change"
    assert np.isnan(kf[0, 0, 4, 7]) and np.isnan(kf[0, 0, 4, 6]), "inf channel and its rotation partner"
    rest = [d for d in range(D) if d not in (6, 7)]
    assert np.all(kf[0, 0, 4, rest] == 0.0), "1/sqrt(inf) = 0 zeroes the other channels"
    assert np.isnan(vf[0, 2, 3, 9]) and v[0, 2, 3, 9] == nan16, "V passes NaN through"
    nanmax = [float(np.nanmax(np.abs(t))) for t in (qf, kf, vf)]
    pbd = _problem(spec, out_kind=1, scale_mode=oracle.SCALE_DYNAMIC)
    am = oracle.amax(pbd, x, inp.wq, inp.wk, inp.pos)
    assert not np.any(np.isnan(am)), am
    assert am.astype(np.float64).tolist() == nanmax, (am, nanmax)
    # an infinite V value: amax inf -> scale = factor = 1 -> inf saturates
    xi = x.copy()
    xi[5, 2 * HD + 1 * D + 3] = inf16
    xi[6, 2 * HD + 3 * D + 0] = _bf16_code(-np.inf)
    xi[7, 2 * HD + 0 * D + 4] = _bf16_code(300.0)
    am_i = oracle.amax(pbd, xi, inp.wq, inp.wk, inp.pos)
    assert am_i[2] == np.inf and am_i[0] == am[0] and am_i[1] == am[1], am_i
    q8, k8, v8, sc = oracle.prepare(pbd, xi, inp.wq, inp.wk, inp.pos)
    assert sc[2] == 1.0 and sc[0] == np.float32(am[0]) / np.float32(448.0), sc
    assert v8[0, 1, 5, 3] == 0x7E and v8[0, 3, 6, 0] == 0xFE, (v8[0, 1, 5, 3], v8[0, 3, 6, 0])
    assert (v8[0, 2, 3, 9] & 0x7F) == 0x7F, "NaN must give a NaN code"
    vv = _widen(oracle.prepare(pb16, xi, inp.wq, inp.wk, inp.pos)[2], spec.in_dtype).astype(np.float32)
    fin = np.isfinite(vv)
    ref = torch.from_numpy(vv[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(v8[fin], ref)
    assert np.all((q8[0, 1, 2] & 0x7F) == 0x7F), "the NaN Q head must stay NaN after the cast"
    # the single-tensor path: its amax skips NaN as well
    xt = np.ascontiguousarray(x[:, 2 * HD:3 * HD])
    pbt = oracle.Problem(batch=1, seq=12, heads=H, head_dim=D, rotary_dim=spec.rotary_dim,
                         in_dtype=spec.in_dtype, tensor=True, out_kind=1, scale_mode=1)
    _, scale = oracle.tensor_prepare(pbt, 2, xt, None, inp.pos)
    assert scale == np.float32(np.float32(nanmax[2]) / np.float32(448.0)), (scale, nanmax[2])


PINS += [pin_scales_degenerate, pin_nonfinite_values]
