"""Two copies of libh3qk in one process (for example two builds that
different components load): each must run its own kernels, including the
ones that raise their shared memory limit on first use.  A copy of the built
library is loaded beside the package's and both run a dynamic e4m3 call
whose results must agree byte for byte."""
import os
import shutil

import numpy as np
import pytest

import gpu_util as G
from video_vae_decoder_qkv_gb300 import h3qk, prepare
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_two_copies_in_one_process():
    import torch

    copy_dir = os.path.join(HERE, "_copies")
    os.makedirs(copy_dir, exist_ok=True)
    copy = os.path.join(copy_dir, "libh3qk_copy.so")
    shutil.copyfile(h3qk.LIB_PATH, copy)
    spec = W.BATCHED_FP8.with_(name="two", batch=2)
    dev = G.to_device(G.inputs(spec))
    kw = dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, batch=spec.batch,
              valid_len=spec.valid_len, scale_mode="dynamic", n_axes=spec.n_axes, axis_dims=spec.axis_dims)
    results = []
    original = h3qk.LIB_PATH
    try:
        for path in (original, copy):
            h3qk.LIB_PATH = path
            h3qk._lib = None
            h3qk.lib()
            q, k, v, sc = prepare(*dev, **kw)
            torch.cuda.synchronize()
            results.append([t.view(torch.uint8).cpu().numpy() for t in (q, k, v)] + [sc.cpu().numpy()])
    finally:
        h3qk.LIB_PATH = original
        h3qk._lib = None
        h3qk.lib()
    for a, b in zip(*results):
        assert np.array_equal(a, b)
