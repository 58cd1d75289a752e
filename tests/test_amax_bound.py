"""The amax early-out's two bounds against the oracle's exact outputs (CPU).

The amax pass skips a warp's head rows when a bound on their 16-bit outputs
cannot exceed the largest exact |y| already seen.  Both bounds are evaluated
here the way the kernel evaluates them (lane layout, summation order and
precision of the approximate sum of squares, the pairwise squares), and every
lane's exact outputs from the oracle must stay under them:

  first bound   max|y| <= c inv max|x| max|w| + 2^-23      (c = 1.45 / 1.47 / 1.49)
  second bound  max|y|^2 t <= K2 max_j (z_j^2 + z_{j+1}^2)  (K2 = 1.01 / 1.04 / 1.06 / 1.09)

with t = ss/D + eps from the approximate sum, inv = 1/sqrt(t) and z = x w.
The second bound is the one the kernel takes when a warp holds 8 or more
token rows (head_dim <= 64); the rows here include the cases that come close
to it: a pass-through pair with one dominant channel, bfloat16 partial sums
that round up, wide weight ranges.  The observed ratios must exceed 1 (the
rows reach the region where the margins matter), and on rows built to round
the bfloat16 sum up at every step the second ratio must exceed what its
constant would be without the packed sum's factor.
"""
import numpy as np
import pytest

import oracle

FP16, BF16 = oracle.FP16, oracle.BF16
K1 = {(FP16, 2): 1.45, (BF16, 1): 1.45, (BF16, 2): 1.47, (BF16, 4): 1.49}
K2 = {(FP16, 2): 1.01, (BF16, 1): 1.04, (BF16, 2): 1.06, (BF16, 4): 1.09}
CH = 2


def _round_bf16(v):
    """float64 -> nearest bfloat16 value (ties to even), normal range."""
    m, e = np.frexp(v)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def _widen(codes, dtype):
    if dtype == FP16:
        return codes.view(np.float16).astype(np.float64)
    return (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _lanes(D):
    """Channel lists of the LPR lanes of one head row (CH = 2 chunks each)."""
    chunks = D // 8
    P = 1 << (chunks - 1).bit_length()
    lpr = max(1, P // CH)
    return [[8 * ch + k for ch in (c, c + lpr) if ch < chunks for k in range(8)] for c in range(lpr)]


def _sum_of_squares(x, lanes, dtype):
    """The bound's approximate sum per row: per lane two partial sums (even
    and odd channels) by fused multiply-adds, bfloat16 or binary32, chunk by
    chunk; their binary32 sum; then the xor tree over the lanes (binary32)."""
    part = []
    for chans in lanes:
        ax = np.zeros(x.shape[0])
        ay = np.zeros(x.shape[0])
        for j in range(0, len(chans), 2):
            a, b = x[:, chans[j]], x[:, chans[j + 1]]
            if dtype == BF16:
                ax = _round_bf16(a * a + ax)
                ay = _round_bf16(b * b + ay)
            else:
                ax = np.float32(a * a + ax).astype(np.float64)
                ay = np.float32(b * b + ay).astype(np.float64)
        part.append(np.float32(ax + ay).astype(np.float64))
    o = len(lanes) // 2
    while o >= 1:
        part = [np.float32(part[c] + part[c ^ o]).astype(np.float64) for c in range(len(lanes))]
        o //= 2
    return part[0]


def _rows(dtype, D, R, n, rng):
    """n rows of one head (Q part) mixing the cases described above."""
    x = rng.standard_normal((n, D))
    kind = np.arange(n) % 4
    # 1: a pass-through pair with one dominant channel
    for i in np.nonzero(kind == 1)[0]:
        j = R + 2 * int(rng.integers(0, (D - R) // 2)) if R < D else 2 * int(rng.integers(0, D // 2))
        x[i, j] = rng.choice([-1, 1]) * rng.uniform(4, 30)
        x[i, j + 1] = 0.0
    # 2: values near 1 whose squares round up in a bfloat16 sum
    near = np.nonzero(kind == 2)[0]
    x[near] = 1.0 + rng.integers(64, 128, (near.size, D)) / 128.0
    # 3: magnitudes over several binades
    wide = np.nonzero(kind == 3)[0]
    x[wide] *= 2.0 ** rng.uniform(-6, 6, (wide.size, D))
    conv = oracle.f32_to_f16 if dtype == FP16 else oracle.f32_to_bf16
    return conv(x.astype(np.float32))


@pytest.mark.parametrize("dtype", [FP16, BF16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("D,R", [(16, 12), (32, 24), (64, 48), (128, 96)])
def test_bounds_cover_the_exact_outputs(dtype, D, R):
    rng = np.random.default_rng([D, R, dtype])
    H, n = 2, 3000
    eps = 1e-6
    w = rng.uniform(0.5, 1.5, D).astype(np.float32)
    w[rng.permutation(D)[: D // 4]] *= np.float32(2.0) ** rng.integers(-3, 4, D // 4).astype(np.float32)
    wk = rng.uniform(0.5, 1.5, D).astype(np.float32)
    q16 = _rows(dtype, D, R, n * H, rng).reshape(n, H * D)
    qkv = np.zeros((n, 3 * H * D), np.uint16)
    qkv[:, : H * D] = q16
    qkv[:, H * D: 2 * H * D] = _rows(dtype, D, R, n * H, rng).reshape(n, H * D)
    pos = rng.integers(0, 4096, (n, 1)).astype(np.int32)
    pb = oracle.Problem(batch=1, seq=n, heads=H, head_dim=D, rotary_dim=R, n_axes=1, axis_dims=(R,),
                        in_dtype=dtype, out_kind=oracle.OUT_16B, scale_mode=oracle.SCALE_NONE, valid_len=n,
                        row_stride=3 * H * D, eps=eps, theta=10000.0)
    y16 = oracle.row16(pb, qkv, w, wk, pos, np.arange(n))[0]           # exact Q outputs [n, H, D]
    lanes = _lanes(D)
    r1 = r2 = 0.0
    for h in range(H):
        x = _widen(q16[:, h * D:(h + 1) * D], dtype)
        y = np.abs(_widen(y16[:, h], dtype))
        ss = _sum_of_squares(x, lanes, dtype)
        t = np.float32(np.float32(ss * np.float32(1.0 / D)) + np.float32(eps)).astype(np.float64)
        assert np.all((ss < 2.0 ** 126) & (t >= 2.0 ** -96))       # the guards do not fire here
        inv_lo = (1.0 - 2.0 ** -21) / np.sqrt(t)                   # rsqrtf within 2^-21 relative
        z = np.float32(x * w.astype(np.float64)).astype(np.float64)
        sq = np.float32(z[:, 0::2] ** 2 + np.float32(z[:, 1::2] ** 2).astype(np.float64)).astype(np.float64)
        for chans in lanes:
            ym = y[:, chans].max(axis=1)
            b1 = K1[(dtype, CH)] * inv_lo * np.abs(x[:, chans]).max(axis=1) * np.abs(w[chans]).max() + 2.0 ** -23
            assert np.all(ym <= b1), (h, chans[0], float(np.max(ym / b1)))
            r1 = max(r1, float(np.max((ym - 2.0 ** -23) / (b1 - 2.0 ** -23) * K1[(dtype, CH)])))
            m = sq[:, [c // 2 for c in chans[0::2]]].max(axis=1)
            live = ym >= 2.0 ** -12
            ratio = ym[live] ** 2 * t[live] / m[live]
            assert np.all(ratio <= K2[(dtype, CH)] * (1 - 2.0 ** -20)), (h, chans[0], float(ratio.max()))
            r2 = max(r2, float(ratio.max()))
    # The rows reach the region where the margins matter: a pass-through pair
    # with a dominant channel meets its norm, and the rounding and the
    # approximate sum push the ratio above 1.
    assert r2 > 1.0, r2
    assert r1 > 1.0, r1


_BF16_POS = (np.arange(0x0080, 0x7F80, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _rounding_up(first, steps):
    """bfloat16 values after `first` whose squares, accumulated by bfloat16
    fused multiply-adds, round the running sum up by the most at each step."""
    acc = float(_round_bf16(np.array([first * first]))[0])
    vals = [first]
    for _ in range(steps):
        c = _BF16_POS[(_BF16_POS ** 2 < acc * 2.0 ** -3) & (_BF16_POS ** 2 > acc * 2.0 ** -12)]
        s = acc + c * c
        v = c[int(np.argmax(_round_bf16(s) - s))]
        vals.append(v)
        acc = float(_round_bf16(np.array([acc + v * v]))[0])
    return vals


def test_second_bound_needs_the_packed_sum_factor():
    """Rows built so that the bfloat16 sum of squares rounds up at every step
    and the lane's largest output is a pass-through channel with a zero
    partner (its pair norm is the value itself): the ratio then exceeds what
    the constant would be without the (1 + 2^-8)^(4 CH) factor of the packed
    sum, and stays under the kernel's 1.06."""
    rng = np.random.default_rng(7)
    D, R, n = 64, 16, 64
    even = [16, 18, 20, 22, 48, 50, 52, 54]      # lane 2 of 4 at head_dim 64; rotary 16: all pass-through
    odd = [19, 21, 23, 49, 51, 53, 55]            # channel 17 (the partner of 16) stays 0
    big = _BF16_POS[(_BF16_POS >= 4) & (_BF16_POS < 8)]
    big = big[np.argsort(-_round_bf16(big * big) / (big * big))][:8]
    small = _BF16_POS[(_BF16_POS > 0.5) & (_BF16_POS < 1)]
    x = np.zeros((n, D))
    for i in range(n):
        x[i, even] = _rounding_up(big[i % 8], 7)
        x[i, odd] = _rounding_up(small[int(rng.integers(0, small.size))], 6)
        x[i] *= 2.0 ** int(rng.integers(-2, 3))
    q16 = oracle.f32_to_bf16(x.astype(np.float32)).reshape(n, D)
    assert np.array_equal(_widen(q16, BF16), x)
    qkv = np.zeros((n, 3 * D), np.uint16)
    qkv[:, :D] = q16
    w = np.ones(D, np.float32)
    pos = rng.integers(0, 4096, (n, 1)).astype(np.int32)
    pb = oracle.Problem(batch=1, seq=n, heads=1, head_dim=D, rotary_dim=R, n_axes=1, axis_dims=(R,),
                        in_dtype=BF16, out_kind=oracle.OUT_16B, scale_mode=oracle.SCALE_NONE, valid_len=n,
                        row_stride=3 * D, eps=1e-6, theta=10000.0)
    y = np.abs(_widen(oracle.row16(pb, qkv, w, w, pos, np.arange(n))[0][:, 0], BF16))
    lanes = _lanes(D)
    t = np.float32(np.float32(_sum_of_squares(x, lanes, BF16) * np.float32(1.0 / D)) + np.float32(1e-6))
    sq = np.float32(x[:, 0::2] ** 2 + x[:, 1::2] ** 2).astype(np.float64)
    chans = lanes[2]
    ratio = y[:, chans].max(axis=1) ** 2 * t.astype(np.float64) / sq[:, [c // 2 for c in chans[0::2]]].max(axis=1)
    assert ratio.max() <= K2[(BF16, CH)] * (1 - 2.0 ** -20), ratio.max()
    without_sum_factor = (1 + 2.0 ** -8) ** 4 * (1 + 2.0 ** -9) ** 2 * (1 + 2.0 ** -16)
    assert ratio.max() > without_sum_factor, (ratio.max(), without_sum_factor)
