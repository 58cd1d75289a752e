"""The chained launches of a dynamic call (zero the amax words, the amax pass,
then the cast; the last two as programmatic dependents of the kernel before
them) against the oracle, bit for bit, in the settings where their ordering
matters:
- calls captured in a CUDA graph and replayed, several calls per graph with
  different inputs and one shared workspace;
- a call enqueued right after a device kernel that produces its input on the
  same stream (the call's first kernel is never chained, so it sees the
  finished input);
- calls back to back on one stream with different inputs, shared outputs and
  one workspace, with no synchronisation between them.
"""
import numpy as np
import pytest

import gpu_util as G
from video_vae_decoder_qkv_gb300 import prepare
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SPECS = [W.LATENT_65K_E4M3.with_(name=f"chain{k}", seq=1200, grid=(1, 20, 60), seed=40 + k,
                                 outlier_scale=[50.0, 5.0, 20.0][k]) for k in range(3)]


def _call(dev, outs, sc, ws, spec, stream=None):
    qkv, wq, wk, pos = dev
    prepare(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim,
            valid_len=spec.valid_len, scale_mode="dynamic", n_axes=spec.n_axes, axis_dims=spec.axis_dims,
            out=outs, out_scales=sc, workspace=ws, stream=stream)


def _buffers(spec):
    import torch

    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    outs = tuple(torch.full(shape, 0xA5, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
                 for _ in range(3))
    return outs, torch.zeros(3, dtype=torch.float32, device="cuda")


def _check(spec, inp, outs, sc):
    want = G.oracle_full(inp)
    for name, g, w in zip("qkv", outs, want[:3]):
        G.assert_codes_equal(G.host_codes(g), w, f"{spec.name} {name}")
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), np.asarray(want[3], np.float32).view(np.uint32))


def test_dynamic_calls_in_a_cuda_graph():
    import torch

    inps = [G.inputs(s) if i < 2 else W.generate(s) for i, s in enumerate(SPECS)]
    devs = [G.to_device(inp) for inp in inps]
    bufs = [_buffers(s) for s in SPECS]
    ws = torch.zeros(4, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        for spec, dev, (outs, sc) in zip(SPECS, devs, bufs):   # warm-up outside the capture
            _call(dev, outs, sc, ws, spec, stream=side)
    side.synchronize()
    for outs, sc in bufs:
        for t in outs:
            t.view(torch.uint8).fill_(0xA5)
        sc.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for spec, dev, (outs, sc) in zip(SPECS, devs, bufs):
            _call(dev, outs, sc, ws, spec, stream=side)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for spec, inp, (outs, sc) in zip(SPECS, inps, bufs):
        _check(spec, inp, outs, sc)


def test_dynamic_call_right_after_the_kernel_that_writes_its_input():
    import torch

    spec = SPECS[0]
    inp = G.inputs(spec)
    src, wq, wk, pos = G.to_device(inp)
    qkv = torch.zeros_like(src)
    outs, sc = _buffers(spec)
    ws = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            qkv.zero_()
            qkv.copy_(src)          # a device kernel producing the input on the same stream
            _call((qkv, wq, wk, pos), outs, sc, ws, spec, stream=s)
    s.synchronize()
    _check(spec, inp, outs, sc)


def test_back_to_back_dynamic_calls_share_outputs_and_workspace():
    import torch

    inps = [G.inputs(s) for s in SPECS[:2]]
    devs = [G.to_device(inp) for inp in inps]
    outs, sc = _buffers(SPECS[0])
    ws = torch.zeros(4, dtype=torch.int32, device="cuda")
    # the larger amax first, then the smaller one: the second call must not
    # see the first call's amax words
    for _ in range(3):
        _call(devs[0], outs, sc, ws, SPECS[0])
        _call(devs[1], outs, sc, ws, SPECS[1])
    torch.cuda.synchronize()
    _check(SPECS[1], inps[1], outs, sc)
