"""Host-side logic of bench.py, on CPU: argument contract, byte accounting,
clock parsing, the library's shrink split, and the multi-rank timing
reduction (gloo, world size 2)."""
import os
import socket

import numpy as np
import pytest

import bench


def test_args_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.steps >= 1 and a.warmup >= 3 and a.impl == "ours"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    assert bench.parse_args(["--impl", "reference"]).impl == "reference"


def test_layer_bytes_decode():
    # W0 32 MiB + D (A+B) slices + x + y; ~40.6 MiB at the expected ~30.5
    # distinct adapters of the decode workload
    b = bench.layer_bytes(64, 4096, 4096, 16, 30.5)
    assert abs(b / 2 ** 20 - 40.6) < 0.2
    g = bench.gemm_bytes(64, 4096, 4096)
    assert g < b and g > 32 * 2 ** 20


def _ksplit_cases():
    fixed = [(64, 4096, 1024, 256, 16), (8752, 4096, 1024, 64, 64),
             (8752, 4096, 14336, 64, 64), (9081, 4096, 14336, 64, 64),
             (1000, 200, 20008, 24, 16), (700, 1032, 12296, 24, 64),
             (256, 14336, 1024, 250, 64), (32, 4096, 1024, 1024, 16), (1, 64, 1024, 3, 8),
             # either side of two waves of 256 x 256 tiles (304 on 152 SMs)
             (1024, 512, 256 * 76, 16, 16), (1024, 512, 256 * 76 - 8, 16, 16),
             (257, 512, 256 * 152, 16, 16), (257, 512, 256 * 151, 16, 16),
             (2048, 512, 256 * 38, 16384, 8)]
    rng = np.random.default_rng(20261203)
    drawn = [(int(rng.integers(1, 20000)), 8 * int(rng.integers(1, 2048)),
              8 * int(rng.integers(1, 6000)), int(rng.integers(1, 3000)),
              int(rng.choice([8, 16, 32, 64, 128]))) for _ in range(40)]
    return fixed + drawn


def test_fused_ksplit_matches_library():
    """bench.py sizes its buffers with a mirror of the library's shrink-split
    rule (the folded tensor-core split at rank 64 / 128, split 1 where the
    256 x 256 prefill tiles run); the workspace size the library reports pins
    the mirror on fixed and drawn shapes."""
    from lora_serving_device_gb300 import build, lora as L
    build.build()
    for T, d_in, d_out, n_slots, r in _ksplit_cases():
        ks = bench.fused_ksplit(T, d_in, d_out, n_slots, r)
        cap = min(T, n_slots)
        head = 16 + T * 4 + cap * 4 + (cap + 1) * 4 + 4
        if T > 256:                        # the shrink's fold counters
            head += (-(-T // 128) + cap) * 4
        head = -(-head // 256) * 256
        body = -(-(head + ks * T * r * 4) // 256) * 256
        if T <= 256:                       # decode-sized: split-K fp32 base product
            S = L.lora_decode_split(T, d_in, d_out)
            assert S >= 1
            # one token tile: the split does not depend on T
            assert all(L.lora_decode_split(t, d_in, d_out) == S for t in (1, 33, 129, 256))
            body += S * T * d_out * 4
        want = -(-body // 256) * 256
        assert L.lora_workspace_bytes(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots) == want


def test_graph_chunk_divides_steps_and_fits_warmup():
    for K, W in [(20, 5), (20, 3), (100000, 5000), (7, 3), (1, 3), (13, 13), (600, 1000)]:
        g = bench.graph_chunk(K, W)
        assert K % g == 0 and 1 <= g <= max(1, min(W, K, bench.GRAPH_STEPS))
    assert bench.graph_chunk(20, 5) == 5 and bench.graph_chunk(100000, 5000) == 500


def test_parse_clocks_window():
    lines = [
        "2026/12/02 10:00:00.000, 0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:01.000, 0, 1500, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active",
    ]
    t0 = bench._smi_time("2026/12/02 10:00:00.000")
    s = bench.parse_clocks(lines, (t0 - 0.01, t0 + 0.5))
    assert s["samples"] == 1 and s["sm_mhz"] == 1965 and s["reasons"] == []


def test_parse_clocks():
    lines = [
        "2026/12/02 10:00:00.000, 0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.200, 0, 1980, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.400, 0, 345, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = bench.parse_clocks(lines)
    assert s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert 1965 <= s["sm_mhz"] <= 1980        # idle sample excluded from "under load"
    assert bench.parse_clocks([])["reasons"] == ["unsampled"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch.distributed as dist
    bench.dist_setup("gloo")
    bench.barrier()
    got = bench.reduce_max(10.0 * (rank + 1))
    bench.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_reduce_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 20.0, 1: 20.0}


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1"])) == 0
    assert capsys.readouterr().out == ""


def test_gpus_n_relaunches_under_torch_distributed(monkeypatch):
    """--gpus N > 1 without a launcher re-runs the script with N ranks on this
    node (rendezvous on 127.0.0.1); with a launcher, a different world size is
    refused."""
    calls = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    assert bench.main(["--gpus", "2", "--steps", "3", "--warmup", "3"]) == 0
    cmd = calls[0]
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=2" in cmd and cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-6:] == ["--gpus", "2", "--steps", "3", "--warmup", "3"]
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2", "--steps", "3", "--warmup", "3"])
