"""GPU parity of h3qk_prepare_sage (float32 Q, float32 K * kv_scale,
float16 V * kv_scale) against the CPU oracle, bit for bit, through the C-ABI:
reduced sizes spanning several warps and blocks with a ragged tail, every
lane layout (head_dim 8 ... 256, non-power-of-two chunk counts), both input
types, both output layouts, per-item valid lengths with canaries, V overflow
and subnormal products, non-finite inputs, the empty call, and every element
of the full 65,280-token latent tile in the launch configuration the
benchmark uses."""
import numpy as np
import pytest

import gpu_util as G
import oracle
from video_vae_decoder_qkv_gb300 import prepare_sage
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CANARY_F32 = np.float32(-7.25).view(np.uint32)
CANARY_F16 = 0x5A5A


def _buffers(shape, fill=True):
    import torch

    q = torch.full(shape, -7.25, dtype=torch.float32, device="cuda")
    k = torch.full(shape, -7.25, dtype=torch.float32, device="cuda")
    v = torch.full(shape, CANARY_F16, dtype=torch.int16, device="cuda").view(torch.float16)
    return q, k, v


def _host(q, k, v):
    import torch

    return (q.cpu().numpy().view(np.uint32), k.cpu().numpy().view(np.uint32),
            v.view(torch.int16).cpu().numpy().view(np.uint16))


def _oracle(spec, inp, kvs, layout=0, valid_lens=None, pos=None, threads=G.THREADS):
    pb = G.problem(spec, out_layout=layout, valid_lens=valid_lens)
    shape = ((spec.batch, spec.seq, spec.heads, spec.head_dim) if layout
             else (spec.batch, spec.heads, spec.seq, spec.head_dim))
    out = (np.full(shape, np.float32(-7.25)), np.full(shape, np.float32(-7.25)),
           np.full(shape, CANARY_F16, np.uint16))
    q, k, v = oracle.sage(pb, inp.qkv, inp.wq, inp.wk, inp.pos if pos is None else pos, kv_scale=kvs,
                          out=out, threads=threads)
    return q.view(np.uint32), k.view(np.uint32), v


def _compare(got, want, what, nan=False):
    kinds = ("f32", "f32", "fp16")
    for name, g, w, kind in zip("qkv", got, want, kinds):
        G.assert_codes_equal(g, w, f"{what} {name}", nan_kind=kind if nan else None)


def _run(spec, kvs, layout="head_major", valid_lens=None, dev=None):
    import torch

    inp = G.inputs(spec)
    qkv, wq, wk, pos = dev if dev is not None else G.to_device(inp)
    shape = ((spec.batch, spec.seq, spec.heads, spec.head_dim) if layout == "token_major"
             else (spec.batch, spec.heads, spec.seq, spec.head_dim))
    out = _buffers(shape)
    vl = torch.tensor(valid_lens, dtype=torch.int32, device="cuda") if valid_lens is not None else None
    prepare_sage(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim,
                 kv_scale=kvs, batch=spec.batch, valid_len=spec.valid_len, n_axes=spec.n_axes,
                 axis_dims=spec.axis_dims, theta=spec.theta, eps=spec.eps, out=out, out_layout=layout,
                 valid_lens=vl)
    torch.cuda.synchronize()
    return inp, _host(*out)


SHAPES = {
    # head_dim 128, 24 heads, 3-axis positions: the latent tile's heads
    "latent": W.LATENT_65K.with_(name="s_latent", batch=2, seq=150, grid=(1, 5, 30), valid_len=147),
    # head_dim 64, 16 heads: the decoder tile's heads
    "decoder": W.DECODER_TILE.with_(name="s_dec", seq=330, grid=(2, 11, 15), valid_len=329),
    # 1-D positions, 40 heads x 128
    "prefix": W.PREFIX_104K_STATIC.with_(name="s_prefix", seq=203, valid_len=199, out_kind=W.OUT_16B,
                                         scale_mode=W.SCALE_NONE),
}


@pytest.mark.parametrize("kvs", [1.0, 0.3])
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_sage_matches_oracle(shape, dtype, kvs):
    spec = SHAPES[shape].with_(in_dtype=dtype, out_kind=W.OUT_16B, scale_mode=W.SCALE_NONE)
    inp, got = _run(spec, kvs)
    _compare(got, _oracle(spec, inp, kvs), f"sage {shape} {dtype} {kvs}")


@pytest.mark.parametrize("D,R,dims", [(8, 6, (2, 2, 2)), (16, 12, (4, 4, 4)), (24, 18, (6, 6, 6)),
                                      (64, 0, (0, 0, 0)), (72, 48, (16, 16, 16)), (136, 96, (32, 32, 32)),
                                      (256, 192, (64, 64, 64)), (256, 256, (86, 86, 84))])
def test_sage_head_dims(D, R, dims):
    spec = W.TINY.with_(name=f"s_d{D}", batch=2, seq=70, grid=(2, 5, 7), head_dim=D, rotary_dim=R,
                        axis_dims=dims, heads=5, valid_len=66, in_dtype=W.BF16)
    inp, got = _run(spec, 0.75)
    _compare(got, _oracle(spec, inp, 0.75), f"sage D={D}")


@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_sage_token_major_and_item_lengths(dtype):
    spec = SHAPES["latent"].with_(in_dtype=dtype, batch=4, seq=61, grid=(1, 1, 61), valid_len=61,
                                  out_kind=W.OUT_16B, scale_mode=W.SCALE_NONE)
    lens = (0, 61, 17, 1000)
    inp, got = _run(spec, 0.5, layout="token_major", valid_lens=lens)
    _compare(got, _oracle(spec, inp, 0.5, layout=1, valid_lens=lens), f"sage token-major {dtype}")


@pytest.mark.parametrize("kvs", [3.0e4, 1.0e-6, -2.0, 0.0])
def test_sage_v_overflow_and_subnormal(kvs):
    spec = SHAPES["decoder"].with_(in_dtype=W.BF16, dist="huge", seq=96, grid=(1, 8, 12), valid_len=96)
    inp, got = _run(spec, kvs)
    _compare(got, _oracle(spec, inp, kvs), f"sage kv_scale {kvs}", nan=True)


def test_sage_non_finite_inputs():
    import torch

    spec = SHAPES["decoder"].with_(in_dtype=W.FP16, seq=64, grid=(1, 8, 8), valid_len=64)
    inp = G.inputs(spec)
    qkv = inp.qkv.copy()
    HD = spec.hd
    qkv[3, 5] = 0x7C00          # +inf in a Q head
    qkv[9, HD + 70] = 0x7E00    # NaN in a K head
    qkv[17, 2 * HD + 3] = 0xFC00  # -inf in V
    inp2 = W.Inputs(spec, qkv, inp.wq, inp.wk, inp.pos, inp.static_scales, inp.outlier_cols)
    dev = G.to_device(inp2)
    _, got = _run(spec, 1.0, dev=dev)
    torch.cuda.synchronize()
    _compare(got, _oracle(spec, inp2, 1.0), "sage non-finite", nan=True)


def test_sage_empty_and_no_valid_rows():
    import torch

    H, D = 4, 64
    x = torch.zeros((0, 3 * H * D), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(D, dtype=torch.float32, device="cuda")
    pos = torch.zeros((0, 3), dtype=torch.int32, device="cuda")
    q, k, v = prepare_sage(x, w, w, pos, heads=H, head_dim=D, rotary_dim=48)
    assert q.numel() == 0 and v.dtype == torch.float16
    spec = SHAPES["decoder"].with_(seq=40, grid=(1, 5, 8), valid_len=0)
    inp, got = _run(spec, 1.0)
    assert np.all(got[0] == CANARY_F32) and np.all(got[1] == CANARY_F32) and np.all(got[2] == CANARY_F16)


def test_sage_full_size_bit_exact():
    """The whole 65,280-token latent tile in the benchmark's launch
    configuration: every element of Q, K and V against the oracle run over
    all host cores."""
    import torch

    spec = W.LATENT_65K
    inp = G.inputs(spec)
    dev = G.to_device(inp)
    _, got = _run(spec, 0.25, dev=dev)
    del dev
    torch.cuda.empty_cache()
    _compare(got, _oracle(spec, inp, 0.25), "sage full size")
