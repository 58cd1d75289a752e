"""GPU parity of the call options and of the single-tensor entry point, each
against the CPU oracle byte for byte, through the C-ABI:

- token-major [B, S, H, D] output (the layout cuDNN reads) in every mode;
- per-item valid lengths (valid_lens), including 0, S and out-of-range
  values, with canaries past each item's prefix;
- e4m3 saturation counters (the calibration log of clipped elements);
- h3qk_norm_rope_tensor on one [B, S, H, D] tensor: Q and K (norm + RoPE),
  V (identity, no weight), 16-bit and e4m3 with its own descale.
"""
import numpy as np
import pytest

import gpu_util as G
import oracle
from video_vae_decoder_qkv_gb300 import norm_rope_tensor, prepare
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MODES = {"16b": {}, "dynamic": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC),
         "static": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC)}
SNAME = {W.SCALE_NONE: "none", W.SCALE_DYNAMIC: "dynamic", W.SCALE_STATIC: "static"}


def _dev_out(shape, e4m3, dt, fill):
    import torch

    if e4m3:
        return torch.full(shape, fill & 0xFF, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    f = fill & 0xFFFF
    return torch.full(shape, f - 0x10000 if f >= 0x8000 else f, dtype=torch.int16, device="cuda").view(dt)


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_token_major_output(mode, dtype):
    import torch

    spec = W.LATENT_65K.with_(name="tm", batch=2, seq=150, grid=(1, 5, 30), valid_len=147, in_dtype=dtype,
                              **MODES[mode])
    inp = G.inputs(spec)
    qkv, wq, wk, pos = G.to_device(inp)
    e4m3 = spec.out_kind == W.OUT_E4M3
    dt = torch.float16 if dtype == W.FP16 else torch.bfloat16
    fill = 0xA5 if e4m3 else 0x7D3B
    shape = (spec.batch, spec.seq, spec.heads, spec.head_dim)
    out = tuple(_dev_out(shape, e4m3, dt, fill) for _ in range(3))
    st = torch.from_numpy(inp.static_scales).cuda() if mode == "static" else None
    q, k, v, sc = prepare(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim,
                          rotary_dim=spec.rotary_dim, batch=spec.batch, valid_len=spec.valid_len,
                          scale_mode=SNAME[spec.scale_mode], axis_dims=spec.axis_dims, static_scales=st,
                          out=out, out_layout="token_major")
    kw = {"static_scales": tuple(float(x) for x in inp.static_scales)} if mode == "static" else {}
    pb = G.problem(spec, out_layout=1, **kw)
    odt = np.uint8 if e4m3 else np.uint16
    want = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos,
                          out=tuple(np.full(shape, fill, odt) for _ in range(3)), threads=G.THREADS)
    for name, g, w in zip("qkv", (q, k, v), want[:3]):
        G.assert_codes_equal(G.host_codes(g), w, f"token-major {mode} {name}")
    if e4m3:
        assert np.array_equal(sc.cpu().numpy(), want[3])


@pytest.mark.parametrize("mode", list(MODES))
def test_per_item_valid_lengths(mode):
    import torch

    spec = W.BATCHED_FP8.with_(name="vl", batch=4, seq=61, grid=(1, 1, 61), **MODES[mode]) \
        if mode != "16b" else W.BATCHED_FP8.with_(name="vl", batch=4, seq=61, grid=(1, 1, 61),
                                                  out_kind=W.OUT_16B, scale_mode=W.SCALE_NONE)
    lens = (0, 61, 17, 1000)
    inp = G.inputs(spec)
    qkv, wq, wk, pos = G.to_device(inp)
    e4m3 = spec.out_kind == W.OUT_E4M3
    fill = 0xA5 if e4m3 else 0x7D3B
    out = G.out_tensors(spec, fill=fill)
    st = torch.from_numpy(inp.static_scales).cuda() if mode == "static" else None
    vl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q, k, v, sc = prepare(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim,
                          rotary_dim=spec.rotary_dim, batch=spec.batch, scale_mode=SNAME[spec.scale_mode],
                          axis_dims=spec.axis_dims, static_scales=st, out=out, valid_lens=vl)
    kw = {"static_scales": tuple(float(x) for x in inp.static_scales)} if mode == "static" else {}
    pb = G.problem(spec, valid_lens=lens, **kw)
    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    odt = np.uint8 if e4m3 else np.uint16
    want = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos,
                          out=tuple(np.full(shape, fill, odt) for _ in range(3)), threads=G.THREADS)
    for name, g, w in zip("qkv", (q, k, v), want[:3]):
        G.assert_codes_equal(G.host_codes(g), w, f"valid_lens {mode} {name}")
    if e4m3:
        assert np.array_equal(sc.cpu().numpy(), want[3])


CANARY8 = 0xA5     # e4m3 output fill: padded rows must keep it
SAT_GEOMETRIES = {
    "d64_bf16": W.BATCHED_FP8.with_(name="sat", batch=2, seq=306, grid=(1, 18, 17), valid_len=300),
    "d128_fp16": W.LATENT_65K.with_(name="sat128", batch=2, seq=131, grid=(1, 1, 131), valid_len=127,
                                    in_dtype=W.FP16),
    # 2,560 row groups of 4 tokens: above the small-call threshold, so the
    # unsliced counting instance runs
    "d128_bf16_plain": W.LATENT_65K.with_(name="sat128p", seq=10240, grid=(5, 32, 64), valid_len=10200),
}


@pytest.mark.parametrize("geometry", list(SAT_GEOMETRIES))
@pytest.mark.parametrize("scales", [None, (0.01, 0.02, 0.05), (1e-30, 1.0, 1e30)])
def test_saturation_counts(scales, geometry):
    """A cast with sat_counts runs its own kernel instance: its counts, and
    its codes and scales, must equal the oracle's."""
    import torch

    mode = "dynamic" if scales is None else "static"
    spec = SAT_GEOMETRIES[geometry].with_(**MODES[mode])
    inp = G.inputs(spec)
    qkv, wq, wk, pos = G.to_device(inp)
    counts = torch.zeros(3, dtype=torch.int32, device="cuda")
    st = torch.tensor(scales, dtype=torch.float32, device="cuda") if scales else None
    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    out = tuple(torch.full(shape, CANARY8, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
                for _ in range(3))
    q, k, v, sc = prepare(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim,
                          rotary_dim=spec.rotary_dim, batch=spec.batch, valid_len=spec.valid_len,
                          scale_mode=mode, axis_dims=spec.axis_dims, static_scales=st, sat_counts=counts,
                          out=out)
    torch.cuda.synchronize()
    kw = {"static_scales": tuple(float(x) for x in scales)} if scales else {}
    pb = G.problem(spec, **kw)
    am = oracle.amax(pb, inp.qkv, inp.wq, inp.wk, inp.pos, threads=G.THREADS) if scales is None \
        else np.zeros(3, np.float32)
    _, inv = oracle.scales(pb, am)
    want = oracle.sat_counts(pb, inp.qkv, inp.wq, inp.wk, inp.pos, inv)
    assert counts.cpu().numpy().astype(np.uint32).tolist() == want.tolist()
    full = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos,
                          out=tuple(np.full(shape, CANARY8, np.uint8) for _ in range(3)), threads=G.THREADS)
    for name, g, w in zip("qkv", (q, k, v), full[:3]):
        G.assert_codes_equal(G.host_codes(g), w, f"counted cast {geometry} {mode} {name}", nan_kind="e4m3")
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), full[3].view(np.uint32))


@pytest.mark.parametrize("kind", ["q", "k", "v"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_single_tensor(kind, mode, dtype):
    import torch

    spec = W.PREFIX_104K_STATIC.with_(name="tensor", batch=2, seq=203, valid_len=199, in_dtype=dtype,
                                      **(MODES[mode] if mode != "16b" else dict(out_kind=W.OUT_16B,
                                                                               scale_mode=W.SCALE_NONE)))
    inp = G.inputs(spec)
    t = "qkv".index(kind)
    HD = spec.hd
    x_np = np.ascontiguousarray(inp.qkv[:, t * HD:(t + 1) * HD])
    w_np = (inp.wq, inp.wk, None)[t]
    dt = torch.float16 if dtype == W.FP16 else torch.bfloat16
    x = torch.from_numpy(x_np.view(np.int16)).cuda().view(dt)
    w = torch.from_numpy(w_np).cuda() if w_np is not None else None
    pos = torch.from_numpy(inp.pos).cuda()
    e4m3 = spec.out_kind == W.OUT_E4M3
    fill = 0xA5 if e4m3 else 0x7D3B
    shape = (spec.batch, spec.seq, spec.heads, spec.head_dim)
    out = _dev_out(shape, e4m3, dt, fill)
    st = torch.tensor([inp.static_scales[t]], dtype=torch.float32, device="cuda") if mode == "static" else None
    got, sc = norm_rope_tensor(x, w, pos, kind=kind, heads=spec.heads, head_dim=spec.head_dim,
                               rotary_dim=spec.rotary_dim, batch=spec.batch, valid_len=spec.valid_len,
                               scale_mode=SNAME[spec.scale_mode], n_axes=spec.n_axes, static_scale=st, out=out)
    kw = {"static_scales": (float(inp.static_scales[t]),) * 3} if mode == "static" else {}
    pb = oracle.Problem(batch=spec.batch, seq=spec.seq, heads=spec.heads, head_dim=spec.head_dim,
                        rotary_dim=spec.rotary_dim, n_axes=spec.n_axes, in_dtype=dtype,
                        out_kind=spec.out_kind, scale_mode=spec.scale_mode, valid_len=spec.valid_len,
                        tensor=True, **kw)
    odt = np.uint8 if e4m3 else np.uint16
    want, wsc = oracle.tensor_prepare(pb, t, x_np, w_np, inp.pos, out=np.full(shape, fill, odt),
                                      threads=G.THREADS)
    G.assert_codes_equal(G.host_codes(got), want, f"tensor {kind} {mode}")
    if e4m3:
        assert np.array_equal(sc.cpu().numpy(), np.array([wsc], np.float32))


def test_single_tensor_empty_and_v_without_weight():
    import torch

    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((0, 3), dtype=torch.int32, device="cuda")
    out, sc = norm_rope_tensor(x, None, pos, kind="v", heads=4, head_dim=64, rotary_dim=48,
                               scale_mode="dynamic")
    torch.cuda.synchronize()
    assert out.numel() == 0 and sc.cpu().tolist() == [1.0]
