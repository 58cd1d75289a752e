"""h3qk_prepare_host (host buffers, chunked transfers overlapped with the
kernels) against h3qk_prepare on the same data, byte for byte, through the
C-ABI: several chunks per item with a ragged last chunk, both layouts, all
output modes, per-item valid lengths from a host array, canaries in the
host outputs past each valid prefix, an empty call, and two calls in a row
on one workspace."""
import numpy as np
import pytest

import gpu_util as G
import oracle
from video_vae_decoder_qkv_gb300 import h3qk, prepare, prepare_host
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MODES = {"16b": (W.OUT_16B, W.SCALE_NONE, "none"), "dynamic": (W.OUT_E4M3, W.SCALE_DYNAMIC, "dynamic"),
         "static": (W.OUT_E4M3, W.SCALE_STATIC, "static")}
FILL16, FILL8 = 0x7D3B, 0xA5


def _spec(dtype, mode, **kw):
    ok, sm, _ = MODES[mode]
    d = dict(name="host", batch=2, seq=20000, grid=None, heads=4, head_dim=64, rotary_dim=48, valid_len=19990,
             in_dtype=dtype, out_kind=ok, scale_mode=sm, outlier_frac=0.001, outlier_scale=30.0)
    d.update(kw)
    return W.DECODER_TILE.with_(**d)


def _host_tensors(inp):
    import torch

    dt = torch.float16 if inp.spec.in_dtype == W.FP16 else torch.bfloat16
    qkv = torch.from_numpy(inp.qkv.view(np.int16)).view(dt).pin_memory()
    return (qkv, torch.from_numpy(inp.wq).pin_memory(), torch.from_numpy(inp.wk).pin_memory(),
            torch.from_numpy(inp.pos).pin_memory())


def _outs(spec, layout, device):
    import torch

    shape = ((spec.batch, spec.seq, spec.heads, spec.head_dim) if layout == "token_major"
             else (spec.batch, spec.heads, spec.seq, spec.head_dim))
    if spec.out_kind == W.OUT_E4M3:
        make = lambda: torch.full(shape, FILL8, dtype=torch.uint8)  # noqa: E731
    else:
        make = lambda: torch.full(shape, FILL16 - 0x10000 if FILL16 >= 0x8000 else FILL16,  # noqa: E731
                                  dtype=torch.int16)
    outs = [make() for _ in range(3)]
    if device:
        outs = [t.cuda() for t in outs]
    else:
        outs = [t.pin_memory() for t in outs]
    if spec.out_kind != W.OUT_E4M3:
        dt = torch.float16 if spec.in_dtype == W.FP16 else torch.bfloat16
        outs = [t.view(dt) for t in outs]
    elif device:
        outs = [t.view(torch.float8_e4m3fn) for t in outs]
    return tuple(outs)


def _run_both(spec, layout="head_major", valid_lens=None):
    import torch

    inp = G.inputs(spec)
    mode = MODES[[k for k, v in MODES.items() if v[:2] == (spec.out_kind, spec.scale_mode)][0]][2]
    kw = dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, batch=spec.batch,
              valid_len=spec.valid_len, scale_mode=mode, n_axes=spec.n_axes, axis_dims=spec.axis_dims,
              out_layout=layout)
    st_h = torch.from_numpy(inp.static_scales) if mode == "static" else None
    vl_h = torch.tensor(valid_lens, dtype=torch.int32) if valid_lens is not None else None
    hq = _host_tensors(inp)
    got = prepare_host(*hq, out=_outs(spec, layout, False), static_scales=st_h, valid_lens=vl_h, **kw)
    dev = G.to_device(inp)
    want = prepare(*dev, out=_outs(spec, layout, True),
                   static_scales=st_h.cuda() if st_h is not None else None,
                   valid_lens=vl_h.cuda() if vl_h is not None else None, **kw)
    torch.cuda.synchronize()
    return inp, got, want


def _codes(t):
    import torch

    if t.element_size() == 1:
        return t.cpu().view(torch.uint8).numpy()
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("layout", ["head_major", "token_major"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_host_entry_matches_device_entry(dtype, mode, layout):
    spec = _spec(dtype, mode)
    _, got, want = _run_both(spec, layout)
    for name, g, w in zip("qkv", got[:3], want[:3]):
        G.assert_codes_equal(_codes(g), _codes(w), f"host {mode} {layout} {name}")
    if want[3] is not None:
        assert np.array_equal(got[3].numpy().view(np.uint32), want[3].cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("mode", list(MODES))
def test_host_entry_per_item_lengths_and_canaries(mode):
    spec = _spec(W.BF16, mode, batch=4, seq=9000, valid_len=9000)
    lens = (0, 9000, 8193, 17)
    inp, got, want = _run_both(spec, valid_lens=lens)
    for name, g, w in zip("qkv", got[:3], want[:3]):
        gc, wc = _codes(g), _codes(w)
        G.assert_codes_equal(gc, wc, f"host lens {mode} {name}")
        fill = FILL8 if spec.out_kind == W.OUT_E4M3 else FILL16
        for b, n in enumerate(lens):
            assert np.all(gc[b, :, n:] == fill), (name, b)


def test_host_entry_small_case_against_oracle():
    spec = _spec(W.BF16, "dynamic", batch=1, seq=300, valid_len=297, heads=3, head_dim=128, rotary_dim=96,
                 outlier_scale=50.0)
    inp, got, _ = _run_both(spec)
    pb = G.problem(spec)
    shape = (1, spec.heads, spec.seq, spec.head_dim)
    want = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos,
                          out=tuple(np.full(shape, FILL8, np.uint8) for _ in range(3)), threads=G.THREADS)
    for name, g, w in zip("qkv", got[:3], want[:3]):
        G.assert_codes_equal(_codes(g), w, f"host oracle {name}")
    assert np.array_equal(got[3].numpy().view(np.uint32), want[3].view(np.uint32))


def test_host_entry_empty_call_and_two_calls_in_a_row():
    import torch

    H, D = 4, 64
    x = torch.zeros((0, 3 * H * D), dtype=torch.bfloat16).pin_memory()
    w = torch.ones(D, dtype=torch.float32).pin_memory()
    pos = torch.zeros((0, 3), dtype=torch.int32).pin_memory()
    _, _, _, sc = prepare_host(x, w, w, pos, heads=H, head_dim=D, rotary_dim=48, scale_mode="dynamic")
    torch.cuda.synchronize()
    assert sc.tolist() == [1.0, 1.0, 1.0]
    # two calls sharing one workspace, ordered on the current stream
    a = _spec(W.BF16, "dynamic", batch=1, seq=17000, valid_len=17000, seed=31)
    b = a.with_(seed=32, outlier_frac=0.0)
    o = h3qk.default_opts()
    o.in_dtype, o.n_axes = h3qk.BF16, 3
    ws = torch.empty(h3qk.host_workspace_bytes(a.rows, a.heads, a.head_dim, h3qk.E4M3, h3qk.SCALE_DYNAMIC, o),
                     dtype=torch.uint8, device="cuda")
    res = []
    for spec in (a, b):
        inp = G.inputs(spec)
        hq = _host_tensors(inp)
        res.append(prepare_host(*hq, heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim,
                                scale_mode="dynamic", axis_dims=spec.axis_dims, workspace=ws))
    torch.cuda.synchronize()
    for spec, r in zip((a, b), res):
        inp = G.inputs(spec)
        dev = G.to_device(inp)
        want = prepare(*dev, heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim,
                       scale_mode="dynamic", axis_dims=spec.axis_dims)
        torch.cuda.synchronize()
        for name, g, w_ in zip("qkv", r[:3], want[:3]):
            G.assert_codes_equal(_codes(g), _codes(w_), f"two calls {spec.seed} {name}")
        assert np.array_equal(r[3].numpy().view(np.uint32), want[3].cpu().numpy().view(np.uint32))
    assert not np.array_equal(res[1][3].numpy(), res[0][3].numpy())   # the second call saw its own data
