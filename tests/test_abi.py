"""The C-ABI library without a GPU: it loads, exports every function that
include/h3qk.h declares, lays out h3qk_opts as the binding does, and rejects
bad arguments on the host before touching CUDA.  The fake addresses below
are never dereferenced: every call here fails a host-side check first."""
import ctypes

import pytest

from video_vae_decoder_qkv_gb300 import h3qk

H, D, R = 4, 64, 48
N = 48
A = 0x10000000          # fake, 256-byte aligned device addresses
QKV, WQ, WK, POS = A, A + 0x1000000, A + 0x1001000, A + 0x1002000
OQ, OK_, OV, SC, TAB, WS = (A + 0x2000000, A + 0x3000000, A + 0x4000000, A + 0x5000000,
                            A + 0x5001000, A + 0x5002000)
VL = A + 0x5003000


@pytest.fixture(scope="module")
def L():
    return h3qk.lib()


@pytest.fixture(autouse=True)
def _fake_addresses_only_without_a_device(request):
    """Calls below pass fake device addresses that must never reach a kernel;
    a case that passed the host checks by mistake would launch on them.  So
    they run only where no GPU exists (where a launch just fails)."""
    if request.node.get_closest_marker("pure_host"):
        return
    import torch

    if torch.cuda.is_available():
        pytest.skip("fake-address ABI checks run only on hosts without a GPU")


@pytest.mark.pure_host
def test_every_declared_symbol_is_exported(L):
    names = h3qk.declared_functions()
    assert "h3qk_prepare" in names and len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


@pytest.mark.pure_host
def test_only_the_c_abi_is_exported(L):
    """The library exports its C-ABI and nothing a second copy of it in the
    same process could bind to: no process-wide unique objects (the dynamic
    linker shares those across copies) and no other functions."""
    import shutil
    import subprocess

    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", h3qk.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout.split("\n")
    syms = [line.split() for line in out if line.strip()]
    unique = [s for s in syms if len(s) == 3 and s[1] == "u"]
    assert not unique, unique[:5]
    funcs = {s[2] for s in syms if len(s) == 3 and s[1] == "T"}
    assert funcs == set(h3qk.declared_functions()), sorted(funcs ^ set(h3qk.declared_functions()))


@pytest.mark.pure_host
def test_opts_layout_and_defaults(L):
    o = h3qk.default_opts()
    assert ctypes.sizeof(h3qk.Opts) == 96
    assert o.out_layout == 0 and not o.valid_lens and not o.sat_counts
    assert o.in_dtype == 0 and o.n_axes == 3 and list(o.axis_dims) == [0, 0, 0]
    assert o.eps == pytest.approx(1e-6, rel=1e-7) and o.batch == 1 and o.qkv_row_stride == 0
    assert o.theta == 10000.0 and not o.static_scales and not o.workspace and o.workspace_bytes == 0
    assert L.h3qk_workspace_bytes() == 16
    assert L.h3qk_version() >= 100


@pytest.mark.pure_host
def test_status_strings(L):
    for s in range(5):
        assert h3qk.status_string(s)
    assert h3qk.status_string(99) == "unknown status"


def call(**kw):
    a = dict(qkv=QKV, norm_wq=WQ, norm_wk=WK, positions=POS, tokens=N, heads=H, head_dim=D,
             rotary_dim=R, valid_len=N, out_dtype=h3qk.BF16, scale_mode=h3qk.SCALE_NONE,
             out_q=OQ, out_k=OK_, out_v=OV, out_scales=None, opts=None, stream=None)
    a.update(kw)
    return h3qk.prepare_ptr(**a)


def opts(**kw):
    o = h3qk.default_opts()
    for k, v in kw.items():
        if k == "axis_dims":
            o.axis_dims = (ctypes.c_int32 * 3)(*v)
        else:
            setattr(o, k, v)
    return o


@pytest.mark.parametrize("kw", [
    dict(qkv=None), dict(norm_wq=None), dict(norm_wk=None), dict(positions=None), dict(out_q=None),
    dict(out_v=None), dict(tokens=-1), dict(heads=0), dict(head_dim=12), dict(head_dim=264),
    dict(head_dim=0), dict(rotary_dim=47), dict(rotary_dim=66), dict(rotary_dim=-2),
    dict(valid_len=N + 1), dict(valid_len=-1), dict(out_dtype=7),
    dict(out_dtype=h3qk.FP16, opts=opts(in_dtype=h3qk.BF16)),
    dict(scale_mode=h3qk.SCALE_DYNAMIC), dict(out_dtype=h3qk.E4M3),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_STATIC, out_scales=SC),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_STATIC, out_scales=None, opts=opts(static_scales=TAB)),
    dict(opts=opts(batch=5)), dict(opts=opts(batch=0)), dict(opts=opts(n_axes=2)),
    dict(opts=opts(axis_dims=(16, 16, 14))), dict(opts=opts(axis_dims=(15, 17, 16))),
    dict(opts=opts(n_axes=1, axis_dims=(24, 24, 0))), dict(rotary_dim=46),
    dict(opts=opts(eps=-1.0)), dict(opts=opts(theta=0.0)), dict(opts=opts(in_dtype=3)),
    dict(opts=opts(qkv_row_stride=3 * H * D - 8)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=WS, workspace_bytes=8)),
])
def test_invalid_arguments(kw):
    assert call(**kw) == h3qk.ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [
    dict(qkv=QKV + 8), dict(out_k=OK_ + 2), dict(norm_wq=WQ + 4), dict(positions=POS + 2),
    dict(opts=opts(qkv_row_stride=3 * H * D + 4)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC + 2,
         opts=opts(workspace=WS, workspace_bytes=16)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=WS + 4, workspace_bytes=16)),
])
def test_misaligned(kw):
    assert call(**kw) == h3qk.ERR_MISALIGNED


@pytest.mark.parametrize("kw", [
    dict(out_k=OQ), dict(out_v=OQ + 256), dict(out_q=QKV), dict(out_q=QKV + 4096),
    dict(out_v=WK), dict(out_q=POS),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_STATIC, out_scales=TAB, opts=opts(static_scales=TAB)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=OQ + 16, workspace_bytes=16)),
    # the workspace is zeroed on the stream: it may not overlap any input
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=QKV + 4096, workspace_bytes=16)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=WQ, workspace_bytes=16)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=POS + 32, workspace_bytes=16)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC, valid_len=N // 2,
         opts=opts(workspace=VL, workspace_bytes=16, valid_lens=VL, batch=2)),
    # the counters are written: not over an input, the table or the workspace
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
         opts=opts(workspace=WS, workspace_bytes=16, sat_counts=WS + 4)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_STATIC, out_scales=SC,
         opts=opts(static_scales=TAB, sat_counts=TAB + 4)),
    dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_STATIC, out_scales=SC,
         opts=opts(static_scales=TAB, sat_counts=QKV + 64)),
])
def test_aliasing_outputs(kw):
    assert call(**kw) == h3qk.ERR_ALIAS


def test_valid_call_without_a_device_reports_cuda_error():
    """On a host with no usable GPU a valid call gets as far as the launch and
    reports H3QK_ERR_CUDA."""
    assert call() == h3qk.ERR_CUDA
    assert h3qk.lib().h3qk_last_cuda_error() != 0


def _split_call(fn, **kw):
    import ctypes as C

    L = h3qk.lib()
    h3qk._split_sigs(L)
    a = dict(qkv=QKV, norm_wq=WQ, norm_wk=WK, positions=POS, tokens=N, heads=H, head_dim=D,
             rotary_dim=R, valid_len=N)
    a.update({k: v for k, v in kw.items() if k in a})
    args = [a["qkv"], a["norm_wq"], a["norm_wk"], a["positions"], a["tokens"], a["heads"], a["head_dim"],
            a["rotary_dim"], a["valid_len"]]
    if fn == "amax":
        return L.h3qk_amax(*args, kw.get("out_amax", SC), None, None)
    return L.h3qk_cast(*args, kw.get("amax", TAB), kw.get("out_q", OQ), kw.get("out_k", OK_),
                       kw.get("out_v", OV), kw.get("out_scales", SC), None, None)


@pytest.mark.parametrize("fn,kw,want", [
    ("amax", dict(out_amax=None), h3qk.ERR_INVALID_ARG),
    ("amax", dict(out_amax=SC + 2), h3qk.ERR_MISALIGNED),
    ("amax", dict(out_amax=QKV + 64), h3qk.ERR_ALIAS),
    ("amax", dict(head_dim=12), h3qk.ERR_INVALID_ARG),
    ("cast", dict(amax=None), h3qk.ERR_INVALID_ARG),
    ("cast", dict(out_scales=None), h3qk.ERR_INVALID_ARG),
    ("cast", dict(out_k=OQ), h3qk.ERR_ALIAS),
    ("cast", dict(out_scales=TAB), h3qk.ERR_ALIAS),
    ("cast", dict(out_q=OQ + 4), h3qk.ERR_MISALIGNED),
    ("cast", dict(valid_len=N + 1), h3qk.ERR_INVALID_ARG),
])
def test_split_entry_points_check_arguments(fn, kw, want):
    assert _split_call(fn, **kw) == want


def _sage(**kw):
    a = dict(qkv=QKV, norm_wq=WQ, norm_wk=WK, positions=POS, tokens=N, heads=H, head_dim=D,
             rotary_dim=R, valid_len=N, kv_scale=1.0, out_q=OQ, out_k=OK_, out_v=OV)
    a.update(kw)
    return h3qk.prepare_sage_ptr(a["qkv"], a["norm_wq"], a["norm_wk"], a["positions"], a["tokens"], a["heads"],
                                 a["head_dim"], a["rotary_dim"], a["valid_len"], a["kv_scale"], a["out_q"],
                                 a["out_k"], a["out_v"], None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(kv_scale=float("nan")), h3qk.ERR_INVALID_ARG),
    (dict(kv_scale=float("inf")), h3qk.ERR_INVALID_ARG),
    (dict(out_v=None), h3qk.ERR_INVALID_ARG),
    (dict(head_dim=12), h3qk.ERR_INVALID_ARG),
    (dict(valid_len=N + 1), h3qk.ERR_INVALID_ARG),
    (dict(out_q=OQ + 8), h3qk.ERR_MISALIGNED),
    (dict(out_v=OV + 2), h3qk.ERR_MISALIGNED),
    (dict(out_k=OQ + N * H * D * 4 - 16), h3qk.ERR_ALIAS),   # K starts inside Q (4-byte elements)
    (dict(out_v=QKV + 16), h3qk.ERR_ALIAS),
    (dict(out_q=WQ), h3qk.ERR_ALIAS),
])
def test_sage_entry_point_checks_arguments(kw, want):
    assert _sage(**kw) == want


def test_sage_valid_call_without_a_device_reports_cuda_error():
    assert _sage() == h3qk.ERR_CUDA


def _host(**kw):
    o = h3qk.default_opts()
    o.in_dtype = h3qk.BF16
    for k in ("sat_counts", "workspace"):
        if k in kw:
            setattr(o, k, kw.pop(k))
    a = dict(qkv=QKV, norm_wq=WQ, norm_wk=WK, positions=POS, tokens=N, heads=H, head_dim=D, rotary_dim=R,
             valid_len=N, out_dtype=h3qk.BF16, scale_mode=h3qk.SCALE_NONE, out_q=OQ, out_k=OK_, out_v=OV,
             out_scales=None, ws=A + 0x6000000, ws_bytes=1 << 30)
    a.update(kw)
    return h3qk.prepare_host_ptr(a["qkv"], a["norm_wq"], a["norm_wk"], a["positions"], a["tokens"], a["heads"],
                                 a["head_dim"], a["rotary_dim"], a["valid_len"], a["out_dtype"], a["scale_mode"],
                                 a["out_q"], a["out_k"], a["out_v"], a["out_scales"], o, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(ws=None), h3qk.ERR_INVALID_ARG),
    (dict(ws=A + 0x6000000 + 64), h3qk.ERR_MISALIGNED),
    (dict(ws_bytes=1024), h3qk.ERR_INVALID_ARG),
    (dict(sat_counts=SC), h3qk.ERR_INVALID_ARG),
    (dict(workspace=WS), h3qk.ERR_INVALID_ARG),
    (dict(head_dim=12), h3qk.ERR_INVALID_ARG),
    (dict(out_dtype=h3qk.FP16), h3qk.ERR_INVALID_ARG),
    (dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC), h3qk.ERR_INVALID_ARG),  # no out_scales
    (dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_STATIC, out_scales=SC), h3qk.ERR_INVALID_ARG),  # no table
    (dict(out_q=None), h3qk.ERR_INVALID_ARG),
    (dict(valid_len=N + 1), h3qk.ERR_INVALID_ARG),
])
def test_host_entry_checks_arguments(kw, want):
    assert _host(**kw) == want


def test_host_entry_valid_call_without_a_device_reports_cuda_error():
    assert _host() == h3qk.ERR_CUDA


@pytest.mark.pure_host
def test_host_workspace_bytes():
    o = h3qk.default_opts()
    small = h3qk.host_workspace_bytes(4896, 16, 64, h3qk.FP16, h3qk.SCALE_NONE, o)
    big = h3qk.host_workspace_bytes(65280, 24, 128, h3qk.BF16, h3qk.SCALE_NONE, o)
    dyn = h3qk.host_workspace_bytes(65280, 24, 128, h3qk.E4M3, h3qk.SCALE_DYNAMIC, o)
    assert 0 < small < big < dyn
    assert h3qk.host_workspace_bytes(10, 16, 64, h3qk.FP16, h3qk.SCALE_NONE, o) % 256 == 0
    assert h3qk.host_workspace_bytes(-1, 16, 64, h3qk.FP16, h3qk.SCALE_NONE, o) == 0


def _vae(fn, **kw):
    L = h3qk.lib()
    if fn == "silu":
        f = L.h3qk_silu_and_mul
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                      ctypes.c_void_p, ctypes.c_void_p]
        a = dict(x=QKV, dtype=h3qk.FP16, rows=10, f=64, stride=0, out=OQ)
        a.update(kw)
        return f(a["x"], a["dtype"], a["rows"], a["f"], a["stride"], a["out"], None)
    f = L.h3qk_scaled_residual
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    a = dict(res=OK_, br=QKV, dtype=h3qk.FP16, sc=WQ, rows=10, C=64, n_sc=64, out=OQ)
    a.update(kw)
    return f(a["res"], a["br"], a["dtype"], a["sc"], a["rows"], a["C"], a["n_sc"], a["out"], None)


@pytest.mark.parametrize("fn,kw,want", [
    ("silu", dict(f=12), h3qk.ERR_INVALID_ARG),
    ("silu", dict(dtype=h3qk.E4M3), h3qk.ERR_INVALID_ARG),
    ("silu", dict(stride=100), h3qk.ERR_INVALID_ARG),
    ("silu", dict(x=None), h3qk.ERR_INVALID_ARG),
    ("silu", dict(stride=132), h3qk.ERR_MISALIGNED),
    ("silu", dict(out=OQ + 8), h3qk.ERR_MISALIGNED),
    ("silu", dict(out=QKV + 256), h3qk.ERR_ALIAS),
    ("res", dict(C=12, n_sc=12), h3qk.ERR_INVALID_ARG),
    ("res", dict(n_sc=3), h3qk.ERR_INVALID_ARG),
    ("res", dict(sc=None), h3qk.ERR_INVALID_ARG),
    ("res", dict(out=OK_ + 64), h3qk.ERR_ALIAS),
    ("res", dict(out=QKV), h3qk.ERR_ALIAS),
    ("res", dict(res=OK_ + 4), h3qk.ERR_MISALIGNED),
])
def test_vae_ops_check_arguments(fn, kw, want):
    assert _vae(fn, **kw) == want


def _tensor_call(**kw):
    """h3qk_norm_rope_tensor on fake addresses (kind Q, e4m3 dynamic)."""
    import ctypes as C

    L = h3qk.lib()
    fn = L.h3qk_norm_rope_tensor
    P, I32, I64 = C.c_void_p, C.c_int32, C.c_int64
    fn.restype = C.c_int
    fn.argtypes = [P, P, P, I64, I32, I32, I32, I64, C.c_int, C.c_int, C.c_int, P, P, C.POINTER(h3qk.Opts), P]
    o = kw.pop("opts")
    a = dict(x=QKV, w=WQ, pos=POS, out=OQ, scale=SC)
    a.update(kw)
    return fn(a["x"], a["w"], a["pos"], N, H, D, R, N, h3qk.TENSOR_Q, h3qk.E4M3, h3qk.SCALE_DYNAMIC,
              a["out"], a["scale"], C.byref(o), None)


@pytest.mark.parametrize("kw,want", [
    (dict(opts=opts(workspace=QKV + 256, workspace_bytes=16)), h3qk.ERR_ALIAS),
    (dict(opts=opts(workspace=WQ + 16, workspace_bytes=16)), h3qk.ERR_ALIAS),
    (dict(opts=opts(workspace=POS, workspace_bytes=16)), h3qk.ERR_ALIAS),
    (dict(opts=opts(workspace=WS, workspace_bytes=16, sat_counts=WS + 8)), h3qk.ERR_ALIAS),
    (dict(opts=opts(workspace=WS, workspace_bytes=16, sat_counts=QKV)), h3qk.ERR_ALIAS),
    (dict(opts=opts(workspace=OQ + 32, workspace_bytes=16)), h3qk.ERR_ALIAS),
    (dict(opts=opts(workspace=WS, workspace_bytes=16)), h3qk.ERR_CUDA),
])
def test_single_tensor_workspace_aliasing(kw, want):
    assert _tensor_call(**kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
          opts=opts(workspace=WS, workspace_bytes=16, sat_counts=WS + 16)), h3qk.ERR_CUDA),
    (dict(out_dtype=h3qk.E4M3, scale_mode=h3qk.SCALE_DYNAMIC, out_scales=SC,
          opts=opts(workspace=WS, workspace_bytes=16)), h3qk.ERR_CUDA),
])
def test_disjoint_workspace_and_counters_pass_the_checks(kw, want):
    """Neighbouring but disjoint scratch buffers pass every host check (the
    call then fails only at the launch, there being no GPU)."""
    assert call(**kw) == want


def test_split_cast_counters_not_over_the_amax():
    import ctypes as C

    L = h3qk.lib()
    h3qk._split_sigs(L)
    o = opts(sat_counts=TAB + 4)
    st = L.h3qk_cast(QKV, WQ, WK, POS, N, H, D, R, N, TAB, OQ, OK_, OV, SC, C.byref(o), None)
    assert st == h3qk.ERR_ALIAS


@pytest.mark.pure_host
def test_release_build_has_no_debug_checks(L):
    import ctypes as C

    assert L.h3qk_debug_checks() == 0
    out = (C.c_uint32 * 4)()
    assert L.h3qk_debug_status(out, 0) == h3qk.ERR_INVALID_ARG
    L.h3qk_debug_limit_outputs(-1)   # no effect in a release build


@pytest.mark.pure_host
def test_debug_build_compiles_and_reports_itself():
    """The debug library (kernels with device-side bounds checks) builds for
    sm_103a and says so; nothing here launches a kernel."""
    from video_vae_decoder_qkv_gb300 import build as B

    D = h3qk.load_library(B.build(debug=True))
    assert D.h3qk_debug_checks() == 1
    assert D.h3qk_version() == h3qk.lib().h3qk_version()
