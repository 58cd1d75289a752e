"""The Python binding refuses caller tensors that do not fit what the library
will read or write through their pointers (CPU: meta tensors carry shapes
and dtypes without memory, and every check runs before a pointer is taken).
"""
import pytest

torch = pytest.importorskip("torch")

from video_vae_decoder_qkv_gb300 import h3qk  # noqa: E402

META = torch.device("meta")
H, D, R, T = 4, 64, 48, 32


def _inputs(dtype=torch.bfloat16, width=3 * H * D):
    qkv = torch.empty((T, width), dtype=dtype, device=META)
    w = torch.empty(D, dtype=torch.float32, device=META)
    pos = torch.empty((T, 3), dtype=torch.int32, device=META)
    return qkv, w, w, pos


def _outs(dtype, n=3, shape=(1, H, T, D)):
    return tuple(torch.empty(shape, dtype=dtype, device=META) for _ in range(n))


KW = dict(heads=H, head_dim=D, rotary_dim=R)


def test_prepare_rejects_a_short_output():
    qkv, wq, wk, pos = _inputs()
    out = _outs(torch.bfloat16)
    short = (out[0], torch.empty((1, H, T - 1, D), dtype=torch.bfloat16, device=META), out[2])
    with pytest.raises(ValueError, match=r"out\[1\] must have"):
        h3qk.prepare(qkv, wq, wk, pos, out=short, **KW)


def test_prepare_rejects_a_wrong_element_size():
    qkv, wq, wk, pos = _inputs()
    with pytest.raises(TypeError, match="1-byte elements"):
        h3qk.prepare(qkv, wq, wk, pos, scale_mode="dynamic", out=_outs(torch.bfloat16), **KW)


def test_prepare_rejects_a_strided_output():
    qkv, wq, wk, pos = _inputs()
    big = torch.empty((1, H, T, 2 * D), dtype=torch.bfloat16, device=META)
    out = (big[..., :D], big[..., D:], _outs(torch.bfloat16, 1)[0])
    with pytest.raises(ValueError, match="contiguous"):
        h3qk.prepare(qkv, wq, wk, pos, out=out, **KW)


def test_prepare_rejects_weights_and_positions_that_do_not_fit():
    qkv, wq, wk, pos = _inputs()
    with pytest.raises(ValueError, match="norm_wk must have 64"):
        h3qk.prepare(qkv, wq, torch.empty(D - 8, dtype=torch.float32, device=META), pos, **KW)
    with pytest.raises(TypeError, match="norm_wq must be"):
        h3qk.prepare(qkv, wq.to(torch.float16), wk, pos, **KW)
    with pytest.raises(ValueError, match="positions must have"):
        h3qk.prepare(qkv, wq, wk, pos[: T - 1], **KW)
    with pytest.raises(TypeError, match="positions must be"):
        h3qk.prepare(qkv, wq, wk, pos.to(torch.int64), **KW)


def test_prepare_rejects_narrow_rows():
    qkv, wq, wk, pos = _inputs(width=3 * H * D - 8)
    with pytest.raises(ValueError, match="rows hold"):
        h3qk.prepare(qkv, wq, wk, pos, **KW)


def test_prepare_rejects_short_tables_and_counters():
    qkv, wq, wk, pos = _inputs()
    out = _outs(torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="static_scales is required"):
        h3qk.prepare(qkv, wq, wk, pos, scale_mode="static", out=out, **KW)
    two = torch.empty(2, dtype=torch.float32, device=META)
    with pytest.raises(ValueError, match="static_scales must have at least 3"):
        h3qk.prepare(qkv, wq, wk, pos, scale_mode="static", static_scales=two, out=out, **KW)
    with pytest.raises(ValueError, match="out_scales must have at least 3"):
        h3qk.prepare(qkv, wq, wk, pos, scale_mode="dynamic", out=out, out_scales=two, **KW)
    with pytest.raises(ValueError, match="sat_counts must have at least 3"):
        h3qk.prepare(qkv, wq, wk, pos, scale_mode="dynamic", out=out,
                     sat_counts=torch.empty(2, dtype=torch.int32, device=META), **KW)
    with pytest.raises(ValueError, match="valid_lens must have 2"):
        q2 = torch.empty((2 * T, 3 * H * D), dtype=torch.bfloat16, device=META)
        p2 = torch.empty((2 * T, 3), dtype=torch.int32, device=META)
        h3qk.prepare(q2, wq, wk, p2, batch=2, valid_lens=torch.empty(3, dtype=torch.int32, device=META), **KW)


def test_sage_rejects_a_half_width_output():
    qkv, wq, wk, pos = _inputs()
    out = (_outs(torch.float32, 1)[0], _outs(torch.float16, 1)[0], _outs(torch.float16, 1)[0])
    with pytest.raises(TypeError, match=r"4-byte elements"):
        h3qk.prepare_sage(qkv, wq, wk, pos, out=out, **KW)


def test_split_passes_reject_short_buffers():
    qkv, wq, wk, pos = _inputs()
    with pytest.raises(ValueError, match="out must have at least 3"):
        h3qk.amax(qkv, wq, wk, pos, out=torch.empty(2, dtype=torch.float32, device=META), **KW)
    with pytest.raises(ValueError, match="amax_t must have at least 3"):
        h3qk.cast(qkv, wq, wk, pos, torch.empty(1, dtype=torch.float32, device=META), **KW)
    out = _outs(torch.float8_e4m3fn)
    short = (out[0], out[1], torch.empty((1, H, T, D - 8), dtype=torch.float8_e4m3fn, device=META))
    with pytest.raises(ValueError, match=r"out\[2\] must have"):
        h3qk.cast(qkv, wq, wk, pos, torch.empty(3, dtype=torch.float32, device=META), out=short, **KW)


def test_single_tensor_and_vae_ops_reject_buffers_that_do_not_fit():
    x = torch.empty((T, H * D), dtype=torch.bfloat16, device=META)
    w = torch.empty(D, dtype=torch.float32, device=META)
    pos = torch.empty((T, 3), dtype=torch.int32, device=META)
    with pytest.raises(ValueError, match="out must have"):
        h3qk.norm_rope_tensor(x, w, pos, kind="q", out=torch.empty((1, T, H, D // 2), dtype=torch.bfloat16,
                                                                    device=META), **KW)
    with pytest.raises(ValueError, match="rows hold"):
        h3qk.norm_rope_tensor(x[:, : H * D - 8], w, pos, kind="k", **KW)
    g = torch.empty((16, 64), dtype=torch.float16, device=META)
    with pytest.raises(ValueError, match="out must have"):
        h3qk.silu_and_mul(g, out=torch.empty((16, 16), dtype=torch.float16, device=META))
    res = torch.empty((16, 32), dtype=torch.float32, device=META)
    br = torch.empty((16, 32), dtype=torch.float16, device=META)
    with pytest.raises(ValueError, match="scale must have 1 or 32"):
        h3qk.scaled_residual(res, br, torch.empty(8, dtype=torch.float32, device=META))
    with pytest.raises(ValueError, match="branch must have"):
        h3qk.scaled_residual(res, br[:8], torch.empty(1, dtype=torch.float32, device=META))
