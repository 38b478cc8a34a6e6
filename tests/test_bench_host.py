"""Host logic of bench.py: the algorithmic byte counts behind the roofline
lines and the validity rule of the committed per-kernel DRAM traffic."""
import json
import os
import shutil

import bench
from kimi_delta_attention_bwd_gb300.inputs import WORKLOADS

TOKEN_HEADS = 16 * 2048 * 8  # the 300M layer shape: B x T x H


def test_step_bytes_of_the_300M_layer():
    # bf16 io, dk 32, dv 64: the forward reads q, k, f, v, b and writes o (2 (3 dk + 2 dv + 1) =
    # 450 B per token-head); the backward reads them and dO and writes five gradients (772 B)
    w = WORKLOADS[bench.STEP_WORKLOAD]
    assert (w.B, w.T, w.H, w.dk, w.dv, w.dtype) == (16, 2048, 8, 32, 64, "bf16")
    assert bench.step_bytes(w) == TOKEN_HEADS * (450 + 772)
    assert bench.step_bytes(w, backward=False) == TOKEN_HEADS * 450


def test_forward_kernels_cover_the_forward_bytes_once():
    w = WORKLOADS[bench.STEP_WORKLOAD]
    assert bench.algorithmic_bytes(w, "fwd_chunk") == TOKEN_HEADS * 322  # q, k, f, v, b
    assert bench.algorithmic_bytes(w, "fwd_state") == TOKEN_HEADS * 128  # o
    assert (bench.algorithmic_bytes(w, "fwd_chunk") + bench.algorithmic_bytes(w, "fwd_state")
            == bench.step_bytes(w, backward=False))


def test_backward_kernels_cover_every_backward_byte():
    # each kernel counts what it must read or write itself, so inputs two kernels need (k, f, dO)
    # count twice; the sum covers the backward's own bytes at least once
    w = WORKLOADS[bench.STEP_WORKLOAD]
    bwd = sum(bench.algorithmic_bytes(w, k) for k in ("bwd_scan", "bwd_grad", "bwd_gate"))
    assert bwd >= bench.step_bytes(w) - bench.step_bytes(w, backward=False)


def test_committed_traffic_is_used_only_on_its_own_sources(tmp_path, monkeypatch):
    committed = json.load(open(os.path.join(bench.PROFILES, "ncu_traffic.json")))
    for e in committed.values():
        assert e["source_files"] == list(bench.TC_SOURCES)
    fake = tmp_path / "profiles"
    fake.mkdir()
    shutil.copy(os.path.join(bench.PROFILES, "ncu_traffic.json"), fake / "ncu_traffic.json")
    monkeypatch.setattr(bench, "PROFILES", str(fake))
    sha = bench.source_sha(bench.TC_SOURCES)
    d = json.load(open(fake / "ncu_traffic.json"))
    d["fwd_chunk"]["source_sha"] = sha
    d["fwd_state"]["source_sha"] = "0" * 16  # taken on other sources
    json.dump(d, open(fake / "ncu_traffic.json", "w"))
    assert bench.ncu_traffic("fwd_chunk") == d["fwd_chunk"]["bytes_per_launch"]
    assert bench.ncu_traffic("fwd_state") is None
    assert bench.ncu_traffic("no_such_kernel") is None
    # the general-path sources are not part of the tensor-core kernels' key
    assert bench.source_sha(bench.TC_SOURCES) != bench.source_sha()
