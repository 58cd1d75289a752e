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


@pytest.mark.parametrize("pattern", ["late_max", "rising", "falling", "near_tie", "uniform"])
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_amax_early_out_is_exact(pattern, dtype):
    """The amax pass skips rows whose bound cannot exceed the running max;
    adversarial orders of magnitudes must still give the exact amax."""
    import torch

    spec = W.LATENT_65K.with_(name="eo", batch=2, seq=257, grid=(1, 1, 257), valid_len=250, in_dtype=dtype,
                              out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC)
    inp = G.inputs(spec)
    vals = (inp.qkv.view(np.float16).astype(np.float32) if dtype == W.FP16
            else (inp.qkv.astype(np.uint32) << 16).view(np.float32)).copy()
    rows = spec.rows
    HD = spec.hd
    if pattern == "late_max":
        vals[1 * spec.seq + 249, 5 * 128 + 17] = 900.0          # last valid row of item 1, Q head 5
        vals[0 * spec.seq + 249, HD + 7 * 128 + 100] = -700.0    # K, pass-through channel
    elif pattern == "rising":
        vals *= np.linspace(0.05, 3.0, rows, dtype=np.float32)[:, None]
    elif pattern == "falling":
        vals *= np.linspace(3.0, 0.05, rows, dtype=np.float32)[:, None]
    elif pattern == "near_tie":
        vals[:, :] = np.float32(1.0)
        vals[137, 3 * 128 + 5] = np.float32(1.0078125)
    conv = oracle.f32_to_f16 if dtype == W.FP16 else oracle.f32_to_bf16
    qkv = conv(vals).reshape(inp.qkv.shape)
    mod = W.Inputs(spec, qkv, inp.wq, inp.wk, inp.pos, inp.static_scales)
    dev = G.to_device(mod)
    a = h3_amax(*dev, **_kw(spec))
    torch.cuda.synchronize()
    ref = oracle.amax(G.problem(spec), qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (a.cpu().numpy(), ref)
