"""prepare_dynamic_sharded's exchange on the CPU: two gloo ranks each own half
of the rows; their amax (computed here by the CPU oracle standing in for the
GPU pass) is all-reduced with MAX, and each rank casts with the shared scales.
The codes of the two ranks together must equal the oracle's unsharded dynamic
cast, and both ranks must report the same descales."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _spec():
    from video_vae_decoder_qkv_gb300 import workloads as W

    return W.BATCHED_FP8.with_(batch=1, seq=96, grid=(1, 8, 12), valid_len=90)


def _problem(spec, **kw):
    import oracle

    return oracle.Problem(batch=1, seq=kw.get("seq", spec.seq), heads=spec.heads, head_dim=spec.head_dim,
                          rotary_dim=spec.rotary_dim, in_dtype=spec.in_dtype, out_kind=spec.out_kind,
                          scale_mode=spec.scale_mode, valid_len=kw.get("valid_len", spec.valid_len))


def _worker(rank, world, port, q):
    sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import oracle
    from video_vae_decoder_qkv_gb300 import h3qk
    from video_vae_decoder_qkv_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = _spec()
    inp = W.generate(spec)
    half = spec.seq // world
    r0, r1 = rank * half, (rank + 1) * half
    vl = max(0, min(half, spec.valid_len - r0))
    rows = inp.qkv[r0:r1]
    pos = inp.pos[r0:r1]
    pb = _problem(spec, seq=half, valid_len=vl)

    def amax_fn(qkv, wq, wk, positions, **kw):
        return torch.from_numpy(oracle.amax(pb, rows, inp.wq, inp.wk, pos).copy())

    def cast_fn(qkv, wq, wk, positions, a, **kw):
        scale, inv = oracle.scales(pb, a.numpy())
        codes = oracle.cast_rows(pb, rows, inp.wq, inp.wk, pos, inv, range(vl))
        return codes, scale

    codes, scale = h3qk.prepare_dynamic_sharded(None, None, None, None, group=dist.group.WORLD,
                                                amax_fn=amax_fn, cast_fn=cast_fn)
    q.put((rank, [c.copy() for c in codes], scale.copy()))
    dist.destroy_process_group()


def test_two_gloo_ranks_share_one_scale():
    sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
    import oracle
    from video_vae_decoder_qkv_gb300 import workloads as W

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(2)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    spec = _spec()
    inp = W.generate(spec)
    pb = _problem(spec)
    full_amax = oracle.amax(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
    scale, inv = oracle.scales(pb, full_amax)
    want = oracle.cast_rows(pb, inp.qkv, inp.wq, inp.wk, inp.pos, inv, range(spec.valid_len))
    assert np.array_equal(res[0][2], scale) and np.array_equal(res[1][2], scale)
    for t in range(3):
        got = np.concatenate([res[0][1][t], res[1][1][t]], axis=0)
        assert np.array_equal(got, want[t])
