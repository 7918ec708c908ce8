"""Host-side pieces of bench.py: byte accounting, the cross-rank timing
reduction (two gloo ranks on the CPU) and the JSON of the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_workload_bytes_match_the_per_element_accounting():
    wb = {name: (e, b, nl) for name, e, b, nl in bench.workload_bytes()}
    n1 = 1 << 20
    assert wb["w1_int8_tensor_fwd"][1] == n1 * 8 + n1 // 8 + 4      # one read of x (on chip), y, mask
    assert wb["w1_ste_bwd"][1] == n1 * 8 + n1 // 8
    n5 = 268_435_456
    assert wb["w5_quant4_double"][1] == n5 * 4 + n5 // 2 + n5 // 64 + 4 * (n5 // 16384)
    total = sum(b for _, b, _ in wb.values())
    assert 4.0e9 < total < 4.2e9
    assert sum(nl for _, _, nl in wb.values()) == 12


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs, units = bench.reduce_max_sum(1.0 + rank, 100.0 * (rank + 1))
    bench.barrier()
    q.put((rank, secs, units))
    dist.destroy_process_group()


def test_reduce_max_sum_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2.0, 300.0), (1, 2.0, 300.0)]


def test_reduce_without_process_group_is_identity():
    assert bench.reduce_max_sum(3.5, 7.0) == (3.5, 7.0)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-fraction", "0.002"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_non_zero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_recorded_traffic_follows_the_source_key(tmp_path, monkeypatch):
    """The DRAM traffic recorded for a kernel is reported only while its
    source and the shared device header hash to the recorded key; an edit to
    either makes it null."""
    import bench

    csrc = tmp_path / "fake_quant_numerics_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "kernels_misc.cu").write_text("// kernel source\n")
    (csrc / "qat_device.cuh").write_text("// device header\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    key = bench.source_key("kernels_misc.cu")
    assert len(key) == 16
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel key bytes\n"
        f"k_q4_quant     {key}  1204138496   # read write algorithmic\n"
        "k_q4_dequant   0000000000000000  1148113664\n")
    assert bench.recorded_traffic("k_q4_quant", "kernels_misc.cu") == 1204138496.0
    assert bench.recorded_traffic("k_q4_dequant", "kernels_misc.cu") is None
    (csrc / "qat_device.cuh").write_text("// device header, edited\n")
    assert bench.recorded_traffic("k_q4_quant", "kernels_misc.cu") is None


def test_all_cores_oracle_driver_reproduces_the_serial_oracle():
    """The all-cores CPU baseline runs the oracle's own functions on pieces of
    each call (per-tensor: parallel statistics, the scale, then the map with
    that scale given); its outputs must equal the serial oracle's bit for bit,
    so the two CPU rows time the same computation."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    from fake_quant_numerics_gb300 import workloads as W

    inputs = bench.oracle_sample(1 / 512)
    x1, g1, w2, a3, w4, g4, x5 = inputs
    keep = {}
    with cf.ThreadPoolExecutor(max_workers=4) as pool:
        bench.oracle_step_parallel(inputs, pool, 7, keep=keep)  # 7 pieces: ragged spans
    y1, m1, s1, dx1 = keep["w1"]
    o1 = oracle.fake_quant_int(x1.numpy(), 1, x1.numel(), 8, 0, 0, want_codes=False)
    assert np.array_equal(y1.view(np.uint32), o1["y"].view(np.uint32))
    assert np.array_equal(m1, o1["mask"]) and s1 == o1["scale"][0]
    assert np.array_equal(dx1.view(np.uint32),
                          oracle.ste_backward(g1.numpy(), o1["mask"]).view(np.uint32))
    r2, c2 = w2.shape
    r4, c4 = w4.shape
    serial_rows = [oracle.fake_quant_int(w2.numpy(), r2, c2, 8, 1, 1),
                   oracle.fake_quant_int(w2.numpy(), r2, c2, 4, 0, 1),
                   oracle.fake_quant_int(W.bf16_bits(w4), r4, c4, 4, 0, 2, 128)]
    for (y, codes, mask, sc, zp), o in zip(keep["rows"], serial_rows):
        assert np.array_equal(y.view(np.uint8), o["y"].view(np.uint8))
        assert np.array_equal(codes.view(np.uint8), o["codes"].view(np.uint8))
        assert np.array_equal(mask, o["mask"])
        assert np.array_equal(sc, o["scale"])
    o4 = serial_rows[2]
    assert np.array_equal(keep["dx4"], oracle.ste_backward(W.bf16_bits(g4), o4["mask"]))
    for (y3, m3, s3), fmt in zip(keep["fp8"], (oracle.E4M3, oracle.E5M2)):
        o3 = oracle.fake_quant_fp8(W.bf16_bits(a3), fmt, want_codes=False)
        assert np.array_equal(y3, o3["y"]) and np.array_equal(m3, o3["mask"])
        assert np.float32(s3) == o3["scale"]
    d5, q5, u5, y5 = keep["w5"]
    o5 = oracle.quant4_double(x5.numpy(), roundtrip=True)
    assert np.array_equal(d5, o5["data"]) and np.array_equal(q5, o5["qscales"])
    assert np.array_equal(u5, o5["super_scales"])
    assert np.array_equal(y5.view(np.uint32), o5["y"].view(np.uint32))
