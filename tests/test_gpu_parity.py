"""Parity of the CUDA path with the CPU oracle: bit-exact Q/K/V codes, e4m3
codes and descales (the fused op must reproduce the unfused definition bit
for bit, as vllm-omni #6607's Operations table requires of its fused Q/K
norm + RoPE).  Every call goes through the C-ABI of libh3qk.so.

- reduced shapes of the five workloads, element by element, sized to span
  many warps and blocks with a ragged tail;
- the five workloads at full size, in the launch configuration the benchmark
  times, element by element;
- the plain (unsliced) kernel instance of every head_dim class, input type
  and mode, element by element;
- edge cases: empty calls, valid_len 0 / 1 / S-1, every head_dim class,
  rotary widths and axis splits, padded row strides, batches with ragged
  items, zero / huge / subnormal / unique-code inputs, non-finite inputs,
  canaries around and inside the outputs, another stream, repeat calls;
- a seeded stress matrix of shapes x seeds x value distributions x modes.
"""
import numpy as np
import pytest

import gpu_util as G
import oracle
from video_vae_decoder_qkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CANARY16 = 0x7D3B   # a finite fp16 / bf16 code no path writes by accident
CANARY8 = 0xA5


def _check_full(spec, inp, q, k, v, sc, want, fill=None, nan_kind=None):
    got = [G.host_codes(t) for t in (q, k, v)]
    kind = nan_kind
    for name, g, w in zip("qkv", got, want[:3]):
        G.assert_codes_equal(g, w, f"{spec.name} {name}", nan_kind=kind)
    if spec.out_kind == W.OUT_E4M3:
        s = sc.cpu().numpy()
        assert np.array_equal(s.view(np.uint32), np.asarray(want[3], np.float32).view(np.uint32)), \
            (s, want[3])
    if fill is not None and spec.valid_len < spec.seq:
        for g in got:
            assert np.all(g[:, :, spec.valid_len:] == fill), "padded rows were written"


REDUCED = [
    W.TINY,
    W.DECODER_TILE.with_(seq=612, grid=(2, 18, 17)),
    W.BATCHED_FP8.with_(batch=3, seq=306, grid=(1, 18, 17)),
    W.LATENT_65K.with_(seq=300, grid=(1, 5, 60)),
    W.LATENT_65K_E4M3.with_(seq=300, grid=(1, 5, 60)),
    W.PREFIX_104K_STATIC.with_(seq=1003, valid_len=999),
    W.PREFIX_104K_DYNAMIC.with_(seq=1003, valid_len=999),
]


@pytest.mark.parametrize("spec", REDUCED, ids=[s.name for s in REDUCED])
def test_reduced_workloads_bit_exact(spec):
    inp = G.inputs(spec)
    fill = CANARY8 if spec.out_kind == W.OUT_E4M3 else CANARY16
    q, k, v, sc = G.gpu_prepare(inp, fill=fill)
    want = G.oracle_full(inp, fill=fill)
    _check_full(spec, inp, q, k, v, sc, want, fill=fill)


FULL = [W.TINY, W.DECODER_TILE, W.BATCHED_FP8, W.LATENT_65K, W.LATENT_65K_E4M3,
        W.PREFIX_104K_STATIC, W.PREFIX_104K_DYNAMIC]


@pytest.mark.parametrize("spec", FULL, ids=[s.name for s in FULL])
def test_full_workloads_bit_exact(spec):
    """Every workload at full size, in the launch configuration the benchmark
    times: every element of Q, K and V, and the descales, against the oracle
    run over all host cores (bit-exact, like torch.equal on whole tensors);
    canaries in the padded rows survive."""
    import torch

    inp = G.inputs(spec)
    fill = CANARY8 if spec.out_kind == W.OUT_E4M3 else CANARY16
    q, k, v, sc = G.gpu_prepare(inp, fill=fill)
    torch.cuda.synchronize()
    want = G.oracle_full(inp, fill=fill)
    _check_full(spec, inp, q, k, v, sc, want, fill=fill)
    del q, k, v, sc, want
    torch.cuda.empty_cache()


def _unsliced_rows(tpw: int) -> int:
    """Token rows whose row groups fill at least 16 warps per SM, so the call
    runs the plain (unsliced) kernel instance the large workloads run, plus a
    ragged tail."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 16 * sms * tpw + 3 * tpw + 1


@pytest.mark.parametrize("head_dim,rotary_dim", [(16, 12), (32, 24), (64, 48), (128, 96), (256, 192)])
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("mode", ["16b", "dynamic", "static", "count"])
def test_unsliced_instances_bit_exact(head_dim, rotary_dim, dtype, mode):
    """The plain kernel instance of every head_dim class, input type and mode
    (the ones the full-size workloads run), element by element: enough rows to
    take the unsliced launch, a ragged last row group and a padded tail."""
    lpr = max(1, (1 << (head_dim // 8 - 1).bit_length()) // 2)
    rows = _unsliced_rows(32 // lpr)
    kw = {"16b": {}, "dynamic": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC),
          "static": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC),
          "count": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC)}[mode]
    spec = W.Spec(f"unsliced{head_dim}", batch=1, seq=rows, heads=3, head_dim=head_dim, rotary_dim=rotary_dim,
                  grid=(1, 1, rows), in_dtype=dtype, valid_len=rows - 5, outlier_frac=0.01,
                  outlier_scale=30.0, seed=head_dim + 7, **kw)
    if mode != "count":
        _roundtrip(spec)
        return
    import torch

    inp = G.inputs(spec)
    counts = torch.zeros(3, dtype=torch.int32, device="cuda")
    q, k, v, sc = G.gpu_prepare(inp, fill=CANARY8, sat_counts=counts)
    want = G.oracle_full(inp, fill=CANARY8)
    _check_full(spec, inp, q, k, v, sc, want, fill=CANARY8)
    _, inv = oracle.scales(G.problem(spec), oracle.amax(G.problem(spec), inp.qkv, inp.wq, inp.wk, inp.pos))
    wc = oracle.sat_counts(G.problem(spec), inp.qkv, inp.wq, inp.wk, inp.pos, inv)
    assert counts.cpu().numpy().astype(np.uint32).tolist() == wc.tolist()


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

BASE = W.TINY.with_(name="edge", seq=75, grid=(3, 5, 5))


def _roundtrip(spec, fill=None, **kw):
    inp = G.inputs(spec)
    if fill is None:
        fill = CANARY8 if spec.out_kind == W.OUT_E4M3 else CANARY16
    q, k, v, sc = G.gpu_prepare(inp, fill=fill, **kw)
    want = G.oracle_full(inp, fill=fill)
    _check_full(spec, inp, q, k, v, sc, want, fill=fill)


@pytest.mark.parametrize("mode", ["16b", "dynamic", "static"])
@pytest.mark.parametrize("valid", [0, 1, 74, 75])
def test_valid_prefix_edges(mode, valid):
    kw = {"16b": {}, "dynamic": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC),
          "static": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC)}[mode]
    _roundtrip(BASE.with_(batch=2, valid_len=valid, in_dtype=W.BF16, **kw))


@pytest.mark.parametrize("head_dim,rotary_dim,n_axes,axis_dims", [
    (8, 8, 1, (8,)), (16, 12, 3, (4, 4, 4)), (24, 18, 3, (6, 6, 6)), (40, 30, 3, (10, 10, 10)),
    (64, 0, 1, (0,)), (64, 64, 1, (64,)), (64, 48, 3, (16, 16, 16)), (64, 44, 3, (10, 24, 10)),
    (128, 96, 3, (32, 32, 32)), (128, 128, 1, (128,)), (136, 136, 1, (136,)),
    (256, 192, 3, (64, 64, 64)), (256, 256, 1, (256,)),
])
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_head_dims_and_rotary_splits(head_dim, rotary_dim, n_axes, axis_dims, dtype):
    spec = W.Spec("dims", batch=2, seq=37, heads=3, head_dim=head_dim, rotary_dim=rotary_dim,
                  n_axes=n_axes, axis_dims=axis_dims, grid=(1, 1, 37) if n_axes == 3 else None,
                  in_dtype=dtype, seed=head_dim)
    _roundtrip(spec)
    _roundtrip(spec.with_(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC))


@pytest.mark.parametrize("dist", ["zeros", "huge", "tiny", "subsq", "unique"])
@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("mode", ["16b", "dynamic", "static"])
def test_value_distributions(dist, dtype, mode):
    kw = {"16b": {}, "dynamic": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC),
          "static": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC)}[mode]
    _roundtrip(BASE.with_(dist=dist, in_dtype=dtype, seed=7, **kw))


def test_padded_row_stride_and_ragged_batch():
    spec = W.LATENT_65K.with_(name="stride", batch=5, seq=7, grid=(1, 1, 7), row_stride=3 * 24 * 128 + 24)
    _roundtrip(spec)
    _roundtrip(spec.with_(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC, valid_len=5))


def test_empty_calls():
    import torch

    from video_vae_decoder_qkv_gb300 import prepare

    for mode in ("none", "dynamic", "static"):
        qkv = torch.zeros((0, 3 * 4 * 64), dtype=torch.bfloat16, device="cuda")
        w = torch.ones(64, device="cuda")
        pos = torch.zeros((0, 3), dtype=torch.int32, device="cuda")
        st = torch.tensor([0.5, 0.25, 0.125], device="cuda")
        q, k, v, sc = prepare(qkv, w, w, pos, heads=4, head_dim=64, rotary_dim=48, scale_mode=mode,
                              static_scales=st if mode == "static" else None)
        torch.cuda.synchronize()
        assert q.numel() == 0
        if mode == "dynamic":
            assert sc.cpu().tolist() == [1.0, 1.0, 1.0]
        if mode == "static":
            assert sc.cpu().tolist() == [0.5, 0.25, 0.125]


def test_static_degenerate_table():
    """Zero, negative, subnormal, infinite and NaN table entries give
    scale = factor = 1."""
    spec = BASE.with_(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC, in_dtype=W.BF16)
    for table in ([0.0, -1.0, 1e-40], [np.inf, np.nan, 0.03]):
        inp = G.inputs(spec)
        q, k, v, sc = G.gpu_prepare(inp, fill=CANARY8, static=table)
        want = G.oracle_full(inp, static=table, fill=CANARY8)
        _check_full(spec, inp, q, k, v, sc, want, fill=CANARY8)


@pytest.mark.parametrize("dtype", [W.FP16, W.BF16])
def test_non_finite_inputs_do_not_trap(dtype):
    """NaN and infinity in a few rows: the call succeeds, rows without them
    match the oracle bit for bit, the others match up to NaN payloads; the
    amax leaves NaN out (one V NaN is the last value of its row)."""
    import torch

    nan, pinf, ninf = (0x7E00, 0x7C00, 0xFC00) if dtype == W.FP16 else (0x7FC0, 0x7F80, 0xFF80)
    for kw in ({}, dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC)):
        spec = BASE.with_(in_dtype=dtype, seed=3, **kw)
        inp = G.inputs(spec)
        qkv = inp.qkv.copy()
        qkv[5, 7] = nan       # NaN in Q of head 0
        qkv[9, 300] = pinf    # +inf in K
        qkv[11, 700] = ninf   # -inf in V
        qkv[13, 3 * spec.hd - 1] = nan  # NaN in V
        qkv[14, 2 * spec.hd + 9] = nan  # NaN in V
        bad = W.Inputs(spec, qkv, inp.wq, inp.wk, inp.pos, inp.static_scales)
        q, k, v, sc = G.gpu_prepare(bad, fill=None)
        torch.cuda.synchronize()
        want = G.oracle_full(bad)
        kind = "e4m3" if spec.out_kind == W.OUT_E4M3 else ("fp16" if dtype == W.FP16 else "bf16")
        for name, g, w in zip("qkv", (q, k, v), want[:3]):
            G.assert_codes_equal(G.host_codes(g), w, f"non-finite {name}", nan_kind=kind)
        if sc is not None:
            assert np.array_equal(sc.cpu().numpy(), want[3])


def test_guard_bytes_around_outputs():
    """Writes stay inside [B, H, S, D]: bytes on either side are untouched."""
    import torch

    from video_vae_decoder_qkv_gb300 import prepare

    spec = BASE.with_(batch=3, seq=21, grid=(1, 3, 7), valid_len=19)
    inp = G.inputs(spec)
    qkv, wq, wk, pos = G.to_device(inp)
    n = spec.batch * spec.heads * spec.seq * spec.head_dim
    guard = 4096
    bufs = [torch.full((n + 2 * guard,), 0x3333, dtype=torch.int16, device="cuda") for _ in range(3)]
    out = tuple(b[guard:guard + n].view(torch.float16).view(spec.batch, spec.heads, spec.seq, spec.head_dim)
                for b in bufs)
    prepare(qkv, wq, wk, pos, heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim,
            batch=spec.batch, valid_len=spec.valid_len, out=out)
    torch.cuda.synchronize()
    for b in bufs:
        h = b.cpu().numpy()
        assert np.all(h[:guard] == 0x3333) and np.all(h[guard + n:] == 0x3333)


def test_other_stream_and_repeat_calls():
    import torch

    spec = W.BATCHED_FP8.with_(batch=2, seq=306, grid=(1, 18, 17))
    inp = G.inputs(spec)
    dev = G.to_device(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = G.gpu_prepare(inp, dev=dev)
        b = G.gpu_prepare(inp, dev=dev)
    s.synchronize()
    for x, y in zip(a, b):
        assert np.array_equal(G.host_codes(x), G.host_codes(y))
    want = G.oracle_full(inp)
    _check_full(spec, inp, *a, want)


def test_launch_counter_counts_kernels():
    from video_vae_decoder_qkv_gb300 import h3qk

    spec = BASE.with_(in_dtype=W.BF16)
    inp = G.inputs(spec)
    for kw, n in (({}, 1), (dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC), 3),
                  (dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC), 1)):
        sp = spec.with_(**kw)
        h3qk.launch_count_reset()
        G.gpu_prepare(W.Inputs(sp, inp.qkv, inp.wq, inp.wk, inp.pos, inp.static_scales))
        assert h3qk.launch_count() == n


def _stress_cases(n=64):
    rng = np.random.default_rng(2024)
    cases = []
    for i in range(n):
        D = int(rng.choice([16, 32, 40, 64, 96, 128, 256]))
        n_axes = int(rng.choice([1, 3]))
        if n_axes == 3:
            w = int(rng.integers(0, D // 6 + 1)) * 2
            dims = (w, w, w)
        else:
            dims = (int(rng.integers(0, D // 2 + 1)) * 2,)
        R = sum(dims)
        B = int(rng.integers(1, 4))
        S = int(rng.integers(1, 90))
        H = int(rng.integers(1, 7))
        mode = ["16b", "dynamic", "static"][i % 3]
        kw = {"16b": {}, "dynamic": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_DYNAMIC),
              "static": dict(out_kind=W.OUT_E4M3, scale_mode=W.SCALE_STATIC)}[mode]
        dist = ["normal", "normal", "huge", "tiny", "zeros", "unique", "subsq"][int(rng.integers(0, 7))]
        cases.append(W.Spec(f"stress{i}", batch=B, seq=S, heads=H, head_dim=D, rotary_dim=R,
                            n_axes=n_axes, axis_dims=dims, grid=(1, 1, S) if n_axes == 3 else None,
                            in_dtype=[W.FP16, W.BF16][i % 2], valid_len=int(rng.integers(0, S + 1)),
                            outlier_frac=0.01, outlier_scale=float(rng.choice([1.0, 30.0, 50.0])),
                            dist=dist, seed=i, theta=float(rng.choice([10000.0, 500.0])),
                            eps=float(rng.choice([1e-6, 1e-5])), **kw))
    return cases


@pytest.mark.parametrize("spec", _stress_cases(), ids=lambda s: s.name)
def test_stress_matrix(spec):
    _roundtrip(spec)
