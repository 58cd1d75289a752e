"""h3qk_prepare_noalloc against h3qk_prepare, through the C-ABI.

The no-allocation entry point exists for callers that cannot allocate device
memory when they call the path, such as an engine plugin that is handed all
its memory up front, or a real-time decode loop with a memory budget fixed at
start-up.  In dynamic e4m3 mode it keeps the amax words in the library's own
fixed scratch array instead of a caller workspace.  This file checks, on two
calls in a row, that its output equals h3qk_prepare's bit for bit (the
tolerance of every parity test here).  The first call has a large amax and the
second a small one, so a second call that saw the first call's amax words
would fail.  The file is named to be collected last and passes alone in a
fresh process as well as after the other tests.
"""
import numpy as np
import pytest

import gpu_util as G
from video_vae_decoder_qkv_gb300 import h3qk
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _call(fn, spec, dev, outs, scales, workspace=None):
    import torch

    qkv, wq, wk, pos = dev
    o = h3qk.default_opts()
    o.in_dtype = spec.in_dtype
    o.n_axes = spec.n_axes
    o.batch = spec.batch
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    st = fn(qkv.data_ptr(), wq.data_ptr(), wk.data_ptr(), pos.data_ptr(), spec.rows, spec.heads,
            spec.head_dim, spec.rotary_dim, spec.valid_len, h3qk.E4M3, h3qk.SCALE_DYNAMIC,
            outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), scales.data_ptr(), o,
            torch.cuda.current_stream().cuda_stream)
    assert st == h3qk.OK, h3qk.status_string(st)


def _buffers(spec):
    import torch

    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    outs = [torch.full(shape, 0xA5, dtype=torch.uint8, device="cuda") for _ in range(3)]
    return outs, torch.zeros(3, dtype=torch.float32, device="cuda")


def test_noalloc_matches_prepare_on_two_calls_in_a_row():
    import torch

    base = W.BATCHED_FP8.with_(name="noalloc", batch=2, seq=306, grid=(1, 18, 17), valid_len=300)
    # call 1: large values (outlier columns x50); call 2: the same draw without
    # outliers, so its amax is smaller than call 1's
    specs = [base.with_(outlier_scale=50.0, seed=21), base.with_(outlier_frac=0.0, seed=22)]
    ws = torch.zeros(4, dtype=torch.int32, device="cuda")
    results = []
    for spec in specs:
        dev = G.to_device(G.inputs(spec))
        want, want_sc = _buffers(spec)
        _call(h3qk.prepare_ptr, spec, dev, want, want_sc, workspace=ws)
        got, got_sc = _buffers(spec)
        _call(h3qk.prepare_noalloc_ptr, spec, dev, got, got_sc)
        torch.cuda.synchronize()
        for name, g, w in zip("qkv", got, want):
            G.assert_codes_equal(g.cpu().numpy(), w.cpu().numpy(), f"noalloc {spec.name} {name}")
        assert np.array_equal(got_sc.cpu().numpy().view(np.uint32), want_sc.cpu().numpy().view(np.uint32))
        results.append(got_sc.cpu().numpy())
    assert results[1][0] < results[0][0], "the second call must have the smaller amax"


def test_noalloc_leaves_device_memory_unchanged():
    """The property the entry point exists for: a dynamic call allocates no
    device memory.  After a warm-up call of the same shape (which may load the
    kernels' code on first use), free device memory is the same before and
    after a call and a synchronize."""
    import torch

    spec = W.BATCHED_FP8.with_(name="noalloc_mem", batch=2, seq=306, grid=(1, 18, 17), valid_len=300, seed=23)
    dev = G.to_device(G.inputs(spec))
    outs, sc = _buffers(spec)
    _call(h3qk.prepare_noalloc_ptr, spec, dev, outs, sc)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        _call(h3qk.prepare_noalloc_ptr, spec, dev, outs, sc)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, (free0, free1)
