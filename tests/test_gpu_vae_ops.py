"""GPU parity of the adjacent decoder-block operations (SwiGLU after the w1
projection, scaled residual) with the CPU oracle, bit for bit, through the
C-ABI: the B300 table's shapes of the vllm-omni operators page (SwiGLU input
[1, 1797, 16384], scaled residual input [2, 1797, 2048]), both 16-bit types,
special values, a padded row stride, a scalar scale and the in-place
residual update."""
import numpy as np
import pytest

import gpu_util as G
import oracle
from video_vae_decoder_qkv_gb300 import scaled_residual, silu_and_mul

pytestmark = pytest.mark.gpu


def _codes(x32, dtype):
    return oracle.f32_to_f16(x32) if dtype == oracle.FP16 else oracle.f32_to_bf16(x32)


def _dev16(codes, dtype):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).cuda()
    return t.view(torch.float16 if dtype == oracle.FP16 else torch.bfloat16)


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
@pytest.mark.parametrize("rows,f,stride", [(1797, 8192, 16384), (37, 24, 56), (3, 8, 16)])
def test_silu_and_mul(dtype, rows, f, stride):
    import torch

    rng = np.random.default_rng(rows + f)
    x32 = (rng.standard_normal(rows * stride) * 4).astype(np.float32)
    special = np.array([0.0, -0.0, 17.5, -17.5, 60.0, -60.0, 88.5, -88.5, 1e-6, -1e-6, 500.0, -500.0],
                       np.float32)
    x32[:special.size] = special
    codes = _codes(x32, dtype).reshape(rows, stride)
    x = _dev16(codes, dtype)[:, :2 * f] if stride != 2 * f else _dev16(codes, dtype)
    out = silu_and_mul(x)
    torch.cuda.synchronize()
    want = oracle.silu_and_mul(codes, f, dtype)
    G.assert_codes_equal(G.host_codes(out), want, f"silu_and_mul {dtype} {rows}x{f}")


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
@pytest.mark.parametrize("per_channel", [True, False])
def test_scaled_residual(dtype, per_channel):
    import torch

    rng = np.random.default_rng(7 + per_channel)
    rows, C = 2 * 1797, 2048
    res = rng.standard_normal((rows, C)).astype(np.float32)
    br = _codes(rng.standard_normal(rows * C).astype(np.float32), dtype).reshape(rows, C)
    sc = (rng.uniform(0.05, 2.0, C if per_channel else 1)).astype(np.float32)
    r_d = torch.from_numpy(res).cuda()
    s_d = torch.from_numpy(sc).cuda()
    out = scaled_residual(r_d, _dev16(br, dtype), s_d)
    torch.cuda.synchronize()
    want = oracle.scaled_residual(res, br, sc, dtype)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))
    # in place: out is the residual
    scaled_residual(r_d, _dev16(br, dtype), s_d, out=r_d)
    torch.cuda.synchronize()
    assert np.array_equal(r_d.cpu().numpy().view(np.uint32), want.view(np.uint32))
