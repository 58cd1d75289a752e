"""The split dynamic passes h3qk_amax / h3qk_cast against h3qk_prepare and
the oracle, through the C-ABI: the amax equals the oracle's, amax then cast
gives the bytes of one DYNAMIC call, and rows split into shards whose amax is
combined (MAX) cast to the bytes of the unsharded call -- the sequence-parallel
use, with the all-reduce done here on one GPU."""
import numpy as np
import pytest

import gpu_util as G
import oracle
from video_vae_decoder_qkv_gb300 import amax as h3_amax
from video_vae_decoder_qkv_gb300 import cast as h3_cast
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SPECS = [
    W.BATCHED_FP8.with_(batch=3, seq=306, grid=(1, 18, 17), valid_len=300),
    W.PREFIX_104K_DYNAMIC.with_(seq=1003, valid_len=999),
    W.TINY.with_(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC),
]


def _kw(spec):
    return dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, batch=spec.batch,
                valid_len=spec.valid_len, n_axes=spec.n_axes, axis_dims=spec.axis_dims, theta=spec.theta,
                eps=spec.eps)


@pytest.mark.parametrize("spec", SPECS, ids=[s.name for s in SPECS])
def test_amax_then_cast_equals_dynamic_prepare(spec):
    import torch

    inp = G.inputs(spec)
    dev = G.to_device(inp)
    want = G.gpu_prepare(inp, dev=dev, fill=0xA5)   # same canary in padded rows as below
    a = h3_amax(*dev, **_kw(spec))
    out = G.out_tensors(spec, fill=0xA5)
    q, k, v, sc = h3_cast(*dev, a, out=out, **_kw(spec))
    torch.cuda.synchronize()
    ref = oracle.amax(G.problem(spec), inp.qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    for name, g, w in zip("qkv", (q, k, v), want[:3]):
        G.assert_codes_equal(G.host_codes(g), G.host_codes(w), f"split {spec.name} {name}")
    assert np.array_equal(sc.cpu().numpy(), want[3].cpu().numpy())


def test_row_shards_with_combined_amax_equal_one_call():
    import torch

    spec = W.PREFIX_104K_DYNAMIC.with_(seq=1003, valid_len=999)
    inp = G.inputs(spec)
    qkv, wq, wk, pos = G.to_device(inp)
    want = G.gpu_prepare(inp, dev=(qkv, wq, wk, pos))
    cut = 512
    shards = [(0, cut, cut), (cut, spec.seq, spec.valid_len - cut)]
    kw = _kw(spec)
    amaxes = []
    for r0, r1, vl in shards:
        amaxes.append(h3_amax(qkv[r0:r1], wq, wk, pos[r0:r1], **{**kw, "valid_len": vl}))
    combined = torch.maximum(amaxes[0], amaxes[1])        # the all-reduce (MAX)
    codes = [[], [], []]
    scales = []
    for r0, r1, vl in shards:
        q, k, v, sc = h3_cast(qkv[r0:r1], wq, wk, pos[r0:r1], combined, **{**kw, "valid_len": vl})
        torch.cuda.synchronize()
        for t, x in enumerate((q, k, v)):
            codes[t].append(G.host_codes(x)[:, :, :vl])
        scales.append(sc.cpu().numpy())
    for t, name in enumerate("qkv"):
        got = np.concatenate(codes[t], axis=2)
        G.assert_codes_equal(got, G.host_codes(want[t])[:, :, :spec.valid_len], f"shards {name}")
    assert np.array_equal(scales[0], scales[1]) and np.array_equal(scales[0], want[3].cpu().numpy())


# Head geometries: 4 token rows per warp (first bound only), 8 and 16 (first
# bound, then the pairwise one).
GEOMETRIES = {"d128": dict(heads=24, head_dim=128, rotary_dim=96, axis_dims=(32, 32, 32)),
              "d64": dict(heads=16, head_dim=64, rotary_dim=48, axis_dims=(16, 16, 16)),
              "d32": dict(heads=8, head_dim=32, rotary_dim=24, axis_dims=(8, 8, 8))}


@pytest.mark.parametrize("geometry", list(GEOMETRIES))
@pytest.mark.parametrize("pattern", ["late_max", "rising", "falling", "near_tie", "pair_tie", "uniform"])
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_amax_early_out_is_exact(pattern, dtype, geometry):
    """The amax pass skips rows whose bound cannot exceed the running max;
    adversarial orders of magnitudes must still give the exact amax."""
    import torch

    spec = W.LATENT_65K.with_(name="eo", batch=2, seq=257, grid=(1, 1, 257), valid_len=250, in_dtype=dtype,
                              out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC, **GEOMETRIES[geometry])
    inp = G.inputs(spec)
    vals = (inp.qkv.view(np.float16).astype(np.float32) if dtype == W.FP16
            else (inp.qkv.astype(np.uint32) << 16).view(np.float32)).copy()
    rows = spec.rows
    HD = spec.hd
    D, R = spec.head_dim, spec.rotary_dim
    if pattern == "late_max":
        vals[1 * spec.seq + 249, 5 * D + 17] = 900.0            # last valid row of item 1, Q head 5
        vals[0 * spec.seq + 249, HD + 7 * D + R + 4] = -700.0   # K, pass-through channel
    elif pattern == "rising":
        vals *= np.linspace(0.05, 3.0, rows, dtype=np.float32)[:, None]
    elif pattern == "falling":
        vals *= np.linspace(3.0, 0.05, rows, dtype=np.float32)[:, None]
    elif pattern == "near_tie":
        vals[:, :] = np.float32(1.0)
        vals[137, 3 * D + 5] = np.float32(1.0078125)
    elif pattern == "pair_tie":
        # flat rows, and in scattered rows one rotated pair (both channels)
        # and one pass-through channel a step above: the pairwise bounds of
        # those rows sit within a rounding of the running max
        vals[:, :] = np.float32(1.0)
        for r, h, j in ((31, 2, 6), (137, 3, 2), (249, 1, 10), (300, 4, R + 2)):
            vals[r, h * D + j] = np.float32(1.0078125)
            if j < R:
                vals[r, h * D + j + 1] = np.float32(1.0078125)
            vals[r, HD + h * D + j] = np.float32(1.0078125)
    conv = oracle.f32_to_f16 if dtype == W.FP16 else oracle.f32_to_bf16
    qkv = conv(vals).reshape(inp.qkv.shape)
    mod = W.Inputs(spec, qkv, inp.wq, inp.wk, inp.pos, inp.static_scales)
    dev = G.to_device(mod)
    a = h3_amax(*dev, **_kw(spec))
    torch.cuda.synchronize()
    ref = oracle.amax(G.problem(spec), qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (a.cpu().numpy(), ref)


def _sumsq_tree(x):
    """Sum of squares of one 128-channel row in the oracle's order (chunks of
    8 left to right, then the halving tree over 16 chunk sums), binary32."""
    f32 = np.float32
    p = []
    for c in range(16):
        acc = f32(x[8 * c] * x[8 * c])
        for k in range(1, 8):
            acc = f32(acc + f32(x[8 * c + k] * x[8 * c + k]))
        p.append(acc)
    o = 8
    while o >= 1:
        for i in range(o):
            p[i] = f32(p[i] + p[i + o])
        o //= 2
    return p[0]


def _sumsq_fused(x):
    """The same sum in the order of the amax pass's bound at head_dim 128 (8
    lanes of two chunks; fused multiply-adds over even and odd channels, one
    add, then three xor-shuffle levels), binary32."""
    f32 = np.float32
    lanes = []
    for c in range(8):
        ax, ay = f32(0), f32(0)
        for ch in (c, c + 8):
            for i in range(4):
                a, b = float(x[8 * ch + 2 * i]), float(x[8 * ch + 2 * i + 1])
                ax = f32(float(ax) + a * a)
                ay = f32(float(ay) + b * b)
        lanes.append(f32(ax + ay))
    for o in (4, 2, 1):
        lanes = [f32(lanes[c] + lanes[c ^ o]) for c in range(8)]
    return lanes[0]


def _overflow_row(seed=0):
    """A bf16 head row whose squares sum to exactly FLT_MAX in the oracle's
    order while the bound's fused order rounds the same sum to infinity:
    3 copies of 2^(52+k), k = 0..11 (squares 2^(104+2k), summing to
    (2^24 - 1) 2^104 = FLT_MAX with no rounding), plus a few elements whose
    squares sit just below half an ulp of FLT_MAX."""
    import warnings

    rng = np.random.default_rng(seed)
    big = [2.0 ** (52 + k) for k in range(12) for _ in range(3)]
    with warnings.catch_warnings(), np.errstate(over="ignore"):
        warnings.simplefilter("ignore")
        for _ in range(20000):
            x = np.zeros(128)
            pos = rng.permutation(128)
            x[pos[:36]] = big
            for j in range(int(rng.integers(2, 6))):
                x[pos[36 + j]] = (int(rng.integers(128, 256)) / 128.0) * 2.0 ** int(rng.integers(49, 51))
            if np.isfinite(_sumsq_tree(x)) and not np.isfinite(_sumsq_fused(x)):
                return x.astype(np.float32)
    raise AssertionError("no near-overflow row found")


def test_amax_bound_near_binary32_overflow():
    """A row whose approximate sum of squares overflows while the exact one
    does not must not be skipped: its exact values (about 5 x the weight)
    are the Q amax here, above every ordinary row, and come after earlier
    rows of the same warp have set a positive running max."""
    import torch

    spec = W.LATENT_65K.with_(name="ovf", batch=1, seq=64, grid=(1, 8, 8), valid_len=64, in_dtype=W.BF16,
                              outlier_frac=0.0, out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC)
    inp = G.inputs(spec)
    vals = (inp.qkv.astype(np.uint32) << 16).view(np.float32).copy()
    base = oracle.amax(G.problem(spec), inp.qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS)
    row = _overflow_row()
    # The skip decision is taken per warp over the 4 token rows it holds at
    # head_dim 128; the other 3 rows get a flat head (small bounds) so that
    # the decision hinges on the near-overflow row's own bound.
    for r, h in ((1, 3), (6, 17), (33, 9)):     # Q heads after head 0 of the same rows
        g0 = r - r % 4
        vals[g0:g0 + 4, h * 128:(h + 1) * 128] = 1.0
        vals[r, h * 128:(h + 1) * 128] = row
    qkv = oracle.f32_to_bf16(vals).reshape(inp.qkv.shape)
    mod = W.Inputs(spec, qkv, inp.wq, inp.wk, inp.pos, inp.static_scales)
    dev = G.to_device(mod)
    a = h3_amax(*dev, **_kw(spec))
    torch.cuda.synchronize()
    ref = oracle.amax(G.problem(spec), qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS)
    assert ref[0] > base[0], (ref, base)     # the near-overflow rows hold the Q amax
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (a.cpu().numpy(), ref)


def test_amax_bound_with_subnormal_squares():
    """eps = 0 and bf16 rows whose squares fall in the binary32 subnormal
    range (random values near 2^-75 ... 2^-72: squares of a fraction to a few
    dozen quanta, where the bound's fused order and the oracle's order round
    differently and the exact path's own mean square is only a few quanta).
    Such rows never take the early-out (their sum under the root is below
    2^-96), so they sit beside flat warp-mates here and the amax, the
    descales and the e4m3 codes of the dynamic call must equal the
    oracle's."""
    import torch

    spec = W.LATENT_65K.with_(name="sub", batch=1, seq=64, grid=(4, 4, 4), valid_len=64, in_dtype=W.BF16,
                              outlier_frac=0.0, eps=0.0, out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC)
    inp = G.inputs(spec)
    vals = (inp.qkv.astype(np.uint32) << 16).view(np.float32).copy()
    rng = np.random.default_rng(4)
    placements = [((17, 3), -75), ((22, 5), -74), ((41, 2), -73), ((46, 14), -72), ((53, 9), -74)]
    for (r, h), e in placements:
        g0 = r - r % 4
        vals[g0:g0 + 4, h * 128:(h + 1) * 128] = 1.0
        mant = 1.0 + rng.integers(0, 128, 128) / 128.0
        expo = e + rng.integers(-1, 1, 128)
        sign = np.where(rng.random(128) < 0.5, -1.0, 1.0)
        vals[r, h * 128:(h + 1) * 128] = (sign * mant * 2.0 ** expo).astype(np.float32)
    qkv = oracle.f32_to_bf16(vals).reshape(inp.qkv.shape)
    mod = W.Inputs(spec, qkv, inp.wq, inp.wk, inp.pos, inp.static_scales)
    dev = G.to_device(mod)
    a = h3_amax(*dev, **_kw(spec))
    torch.cuda.synchronize()
    pb = G.problem(spec)
    ref = oracle.amax(pb, qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (a.cpu().numpy(), ref)
    q, k, v, sc = G.gpu_prepare(mod, dev=dev, fill=0xA5)
    want = oracle.prepare(pb, qkv, inp.wq, inp.wk, inp.pos,
                          out=tuple(np.full((1, spec.heads, spec.seq, spec.head_dim), 0xA5, np.uint8)
                                    for _ in range(3)), threads=G.THREADS)
    for name, g_, w_ in zip("qkv", (q, k, v), want[:3]):
        G.assert_codes_equal(G.host_codes(g_), w_, f"subnormal rows {name}", nan_kind="e4m3")
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), want[3].view(np.uint32))
