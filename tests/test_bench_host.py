"""Host-side checks of bench.py (no GPU): the algorithmic byte and flop counts, the profile
parsing, and the N>1 aggregation on two gloo ranks."""
import os
import shutil

import pytest

import bench
from recurrent_state_update_gb300 import workloads as wl


def test_decode_algorithmic_bytes_per_token_layer():
    # state read + write 2*H*P*N*2, conv state read + write 2*C_d*(W-1)*2, xBC in, z in, dt, y out
    sh = wl.NEMOTRON_H_8B
    assert sh.conv_dim == 10240
    assert bench.DECODE_BYTES_PER_TOKEN_LAYER == 4_194_304 + 122_880 + 20_480 + 16_384 + 512 + 16_384 == 4_370_944
    assert 256 * bench.DECODE_BYTES_PER_TOKEN_LAYER == 1_118_961_664


def test_prefill_flop_count_one_chunk():
    # one full 256-token chunk: C B^T per group (causal half), masked G X, chunk state, C h per head
    L, H, P, N, G = 256, 128, 64, 128, 8
    tri = L * (L + 1) / 2
    want = G * tri * 2 * N + H * (tri * 2 * P + 4 * L * P * N)
    assert bench.prefill_flops([256], 256) == pytest.approx(want)
    assert bench.prefill_flops([300], 256) == pytest.approx(bench.prefill_flops([256], 256) + bench.prefill_flops([44], 256))


def test_profile_traffic_is_dropped_when_the_kernel_source_changed(tmp_path, monkeypatch):
    root = tmp_path
    (root / "profiles").mkdir()
    src = root / "k.cu"
    src.write_text("kernel v1")
    import hashlib
    digest = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    (root / "profiles" / "k.md").write_text(
        f"# k\n\n- source: `k.cu`\n- source_sha256_16: `{digest}`\n- traffic_bytes_per_launch: `1234` (read + write)\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench._profile_traffic("k") == 1234.0
    src.write_text("kernel v2")
    assert bench._profile_traffic("k") is None
    assert bench._profile_traffic("missing") is None


def test_weak_scaling_value():
    assert bench.weak_scaling_gbs(1_000_000_000, 4, 1000.0) == pytest.approx(4.0)


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 7.5][rank]
    got = bench._max_over_ranks(torch, dist, ms, device="cpu")
    with open(os.path.join(out, f"r{rank}"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks(tmp_path):
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"r{r}").read_text()) == 7.5


REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "e2e", "gpu_launches", "cpu_baseline")


def test_emitted_line_keeps_the_contract(capsys):
    """The JSON line bench.py prints carries every key of the benchmark contract, with the
    roofline, end-to-end, clocks and CPU-baseline objects in their documented shapes."""
    import argparse
    import json
    args = argparse.Namespace(steps=100, warmup=5)
    e2e = {"value": 5.8e3, "unit": "GB/s", "ms_per_step": 9.3, "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 2}
    ck = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 20, "reasons": []}
    cpu = {"value": 20.0, "unit": "GB/s", "cores": 16, "kind": "oracle", "sample": "32 rows"}
    bench.emit(args, 1, 48, 9.0, 6.0e3, 1.3e6, 6.0e3, 0.1875, 6795.1, "measured", e2e, ck, None, cpu)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in REQUIRED:
        assert k in line, k
    assert line["config"]["workload"] and line["higher_is_better"] is True and line["scaling"] == "weak"
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert "traffic" in r
    assert set(("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")) <= set(line["e2e"])
    assert set(("sm_mhz", "sm_max_mhz", "reasons")) <= set(line["clocks"])
    assert set(("value", "unit", "cores", "kind", "sample")) <= set(line["cpu_baseline"])


def test_reference_arm_line(monkeypatch, capsys):
    """bench.py --impl reference: the oracle on the host cores, with the decode arm's metric,
    unit and config (plus its sample), and an e2e object with no host-device bytes."""
    import json
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in REQUIRED:
        assert k in line, k
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == bench.decode_config(1, bench.DECODE["layers"])["workload"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_gpus_flag_must_match_the_launched_ranks():
    """--gpus N without N launched ranks is refused instead of silently measuring one GPU."""
    import subprocess
    import sys
    env = dict(os.environ, WORLD_SIZE="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "8", "--impl", "reference"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode != 0
    assert "WORLD_SIZE=1" in r.stderr and "torch.distributed.run" in r.stderr


@pytest.mark.parametrize("layers", [1, 5, 21, 22, 48, 64])
def test_e2e_groups_cover_every_layer_once(layers):
    """The end-to-end pipeline's layer groups add up to the layer count, and the first and last
    groups (whose upload and download are not hidden behind compute) hold one layer each."""
    g = bench.e2e_groups(layers)
    assert sum(g) == layers and min(g) >= 1
    assert g[0] == 1 and g[-1] == 1
    assert max(g) <= 8
