"""The debug build (libh3qk_debug.so: the kernels' device-side bounds checks
compiled in) through the same binding:
- every entry point on valid calls leaves the check status at zero and gives
  the release library's bytes;
- with the output extent narrowed by the test hook, the checks report the
  stores past it (bit 2, a count, the first offset) and skip them, so the
  bytes past the limit keep their canary and the bytes before it are the
  release library's.
The failure is simulated by a narrower extent, not by an access outside a
buffer, so nothing here touches memory it does not own."""
import contextlib
import ctypes

import numpy as np
import pytest

import gpu_util as G
from video_vae_decoder_qkv_gb300 import build as B
from video_vae_decoder_qkv_gb300 import h3qk
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    return h3qk.load_library(B.build(debug=True))


@contextlib.contextmanager
def _using(L):
    saved = h3qk._lib
    h3qk._lib = L
    try:
        yield
    finally:
        h3qk._lib = saved


def _status(L, reset=True):
    out = (ctypes.c_uint32 * 4)()
    assert L.h3qk_debug_status(out, 1 if reset else 0) == h3qk.OK
    first = out[2] | (out[3] << 32)
    return out[0], out[1], first


CASES = [
    W.LATENT_65K.with_(seq=300, grid=(1, 5, 60)),
    W.LATENT_65K_E4M3.with_(seq=300, grid=(1, 5, 60)),
    W.PREFIX_104K_STATIC.with_(seq=1003, valid_len=999),
    W.BATCHED_FP8.with_(batch=3, seq=306, grid=(1, 18, 17)),
    W.DECODER_TILE.with_(seq=612, grid=(2, 18, 17)),
]


@pytest.mark.parametrize("spec", CASES, ids=[s.name for s in CASES])
def test_debug_build_checks_pass_and_match_release(debug_lib, spec):
    import torch

    assert debug_lib.h3qk_debug_checks() == 1
    _status(debug_lib)
    inp = G.inputs(spec)
    fill = 0xA5 if spec.out_kind == W.OUT_E4M3 else 0x7D3B
    want = [G.host_codes(t) for t in G.gpu_prepare(inp, fill=fill)[:3]]
    with _using(debug_lib):
        got = G.gpu_prepare(inp, fill=fill)
        torch.cuda.synchronize()
    assert _status(debug_lib) == (0, 0, 0)
    for g, w in zip(got[:3], want):
        assert np.array_equal(G.host_codes(g), w)


def test_debug_build_sage_split_tensor_host(debug_lib):
    import torch

    from video_vae_decoder_qkv_gb300 import amax, cast, norm_rope_tensor, prepare_host, prepare_sage

    spec = W.LATENT_65K_E4M3.with_(seq=300, grid=(1, 5, 60))
    inp = G.inputs(spec)
    qkv, wq, wk, pos = G.to_device(inp)
    kw = dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, n_axes=3,
              axis_dims=spec.axis_dims)
    _status(debug_lib)
    with _using(debug_lib):
        prepare_sage(qkv, wq, wk, pos, kv_scale=0.5, **kw)
        a = amax(qkv, wq, wk, pos, **kw)
        cast(qkv, wq, wk, pos, a, **kw)
        x = qkv[:, spec.hd:2 * spec.hd]
        norm_rope_tensor(x, wk, pos, kind="k", scale_mode="dynamic", **kw)
        host = qkv.cpu().pin_memory()
        prepare_host(host, wq.cpu(), wk.cpu(), pos.cpu(), scale_mode="dynamic", **kw)
        torch.cuda.synchronize()
    assert _status(debug_lib) == (0, 0, 0)


def test_debug_build_reports_and_skips_stores_past_the_extent(debug_lib):
    import torch

    spec = W.LATENT_65K.with_(seq=300, grid=(1, 5, 60))
    inp = G.inputs(spec)
    n = spec.batch * spec.heads * spec.seq * spec.head_dim
    limit = n // 3 + 8 * 37          # inside head 2's plane, on an 8-element boundary
    want = [G.host_codes(t) for t in G.gpu_prepare(inp, fill=0x7D3B)[:3]]
    _status(debug_lib)
    debug_lib.h3qk_debug_limit_outputs(limit)
    try:
        with _using(debug_lib):
            got = G.gpu_prepare(inp, fill=0x7D3B)
            torch.cuda.synchronize()
    finally:
        debug_lib.h3qk_debug_limit_outputs(-1)
    what, count, first = _status(debug_lib)
    assert what == 2, what                      # output stores only
    assert count == 3 * (n - limit) // 8, count  # every 8-element store past the limit, in Q, K and V
    assert first >= limit + 1, first
    for g, w in zip(got[:3], want):
        h = G.host_codes(g).reshape(-1)
        assert np.array_equal(h[:limit], w.reshape(-1)[:limit])
        assert np.all(h[limit:] == 0x7D3B)
    # the hook is off again: a clean call reports nothing
    with _using(debug_lib):
        G.gpu_prepare(inp, fill=0x7D3B)
        torch.cuda.synchronize()
    assert _status(debug_lib) == (0, 0, 0)
