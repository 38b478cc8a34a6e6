"""Data-parallel sharding on CPU with gloo, world size 2: every rank runs the
oracle on its own documents (no exchange on the data path) and all-reduces
only dA_log / ddt_bias; the result equals the single-process run."""
import math
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from kimi_delta_attention_bwd_gb300.sharding import shard_documents


def _inputs():
    rng = np.random.RandomState(3)
    lens = [37, 1, 64, 0, 90, 12, 55, 8]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N, H, dk, dv = int(cu[-1]), 2, 4, 3
    x = {"q": rng.randn(N, H, dk), "k": rng.randn(N, H, dk), "v": rng.randn(N, H, dv),
         "f": rng.randn(N, H, dk), "b": rng.randn(N, H), "A_log": np.log(rng.uniform(1, 16, H)),
         "dt_bias": rng.uniform(-6, -2, (H, dk)), "cu_seqlens": cu, "scale": 1 / math.sqrt(dk),
         "h0": rng.randn(len(lens), H, dk, dv) * 0.1}
    dO = rng.randn(N, H, dv)
    dhf = rng.randn(len(lens), H, dk, dv)
    return x, dO, dhf


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import oracle
    x, dO, dhf = _inputs()
    lo, hi, t0, t1, local = shard_documents(x["cu_seqlens"], world, rank)
    xs = {k: (v[t0:t1] if k in ("q", "k", "v", "f", "b") else v) for k, v in x.items()}
    xs["cu_seqlens"] = local
    xs["h0"] = x["h0"][lo:hi]
    o, hf = oracle.forward(xs, threads=1)
    g = oracle.backward(xs, dO[t0:t1], dhf[lo:hi], threads=1)
    dA = torch.from_numpy(g["dA_log"].copy())
    dd = torch.from_numpy(g["ddt_bias"].copy())
    dist.all_reduce(dA)
    dist.all_reduce(dd)
    q.put((rank, t0, t1, lo, hi, o, hf, g["dq"], g["dh0"], dA.numpy(), dd.numpy()))
    dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_shards_cover_documents_once():
    cu = np.array([0, 5, 5, 9, 30, 31, 60], dtype=np.int32)
    for world in (1, 2, 3, 4, 8):
        seen = []
        for r in range(world):
            lo, hi, t0, t1, local = shard_documents(cu, world, r)
            assert local[0] == 0 and local[-1] == t1 - t0
            seen += list(range(lo, hi))
        assert seen == list(range(len(cu) - 1))


def test_two_rank_gloo_matches_single_process():
    from oracle import oracle
    oracle.build("f64")
    x, dO, dhf = _inputs()
    o_ref, hf_ref = oracle.forward(x, threads=1)
    g_ref = oracle.backward(x, dO, dhf, threads=1)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t0, t1, lo, hi, o, hf, dq, dh0, dA, dd in res:
        assert np.array_equal(o, o_ref[t0:t1])
        assert np.array_equal(hf, hf_ref[lo:hi])
        assert np.array_equal(dq, g_ref["dq"][t0:t1])
        assert np.array_equal(dh0, g_ref["dh0"][lo:hi])
        np.testing.assert_allclose(dA, g_ref["dA_log"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dd, g_ref["ddt_bias"], rtol=1e-12, atol=1e-14)
