"""The benchmark's multi-process logic on CPU: two gloo ranks aggregate their
timings the way bench.py does under torchrun (max of times, sum of work), and
the reference arm's non-zero ranks do no work."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r = bench.dist_init("gloo")
    assert (w, r) == (world, rank)
    t_max = bench.max_over_ranks(10.0 + rank, w)
    work = bench.sum_over_ranks(100.0 * (rank + 1), w)
    bench.barrier(w)
    out[rank] = (t_max, work)
    torch.distributed.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    for r in range(world):
        assert out[r] == (11.0, 300.0)


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(2.0, 1) == 2.0


def test_reference_arm_nonzero_rank_does_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert rc == 0
    assert capsys.readouterr().out == ""


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_roofline_bounds_and_fractions():
    """bench.roofline: achieved = work / time in the leg's unit, frac = achieved / peak, for
    the three bounds (the fp32 path's ALU peak is derived: 148 x 128 x 2 x 2.032 GHz)."""
    import bench

    class Leg:
        work, unit, kernel, name = 2e12, "TFLOP/s", "prefill_simt_kernel", "nothing"

        def rate(self, work, ms):
            return work / (ms * 1e-3) / 1e12

    peaks = {"bf16_tflops": 1800.0, "hbm_gbs": 6400.0}
    leg = Leg()
    for bound, peak in (("alu", 148 * 128 * 2 * 2.032e9 / 1e12), ("tensor", 1800.0)):
        leg.bound = bound
        r = bench.roofline(leg, 2.0, peaks, "measured")
        assert r["bound"] == bound and r["unit"] == "TFLOP/s"
        assert abs(r["achieved"] - 1000.0) < 1e-9 and abs(r["peak"] - peak) < 1e-9
        assert abs(r["frac"] - 1000.0 / peak) < 1e-12
    leg.bound, leg.unit = "hbm", "GB/s"
    leg.rate = lambda work, ms: work / (ms * 1e-3) / 1e9
    r = bench.roofline(leg, 2.0, peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - 1e6 / 6400.0) < 1e-9


def test_kernel_fingerprint_ignores_comments_only():
    """A comment-only edit keeps a kernel's source fingerprint (the committed ncu traffic
    still applies); a code edit changes it."""
    import bench
    base = {"prefill_tc.cuh": b"int f() {\n  return 1;  // one\n}\n", "ptx.cuh": b"/* x */ int g;\n"}

    def reader(files):
        return lambda name: files[name]

    fp = bench.kernel_fingerprint("prefill_tc_kernel", reader(base))
    commented = dict(base, **{"prefill_tc.cuh": b"// header\nint f() {\n\n  return 1;\n}\n"})
    assert bench.kernel_fingerprint("prefill_tc_kernel", reader(commented)) == fp
    edited = dict(base, **{"prefill_tc.cuh": b"int f() {\n  return 2;\n}\n"})
    assert bench.kernel_fingerprint("prefill_tc_kernel", reader(edited)) != fp


@pytest.mark.parametrize("name,batch,cfg_key,unit", [
    ("single_head_f32", None, "prefill", "TFLOP/s"),
    ("decode_paged_int8_b64", 2, "decode_int8", "GB/s"),
])
def test_reference_arm_prints_one_contract_line(name, batch, cfg_key, unit):
    """`bench.py --impl reference` (the fp64 oracle on the host cores) prints one JSON line
    with the keys and types the benchmark contract names, on the same metric as our arm
    (a prefill workload, and a decode one with its batch cut to 2 sequences)."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
           "--workload", name, "--steps", "3", "--warmup", "3", "--ref-seconds", "1"]
    if batch is not None:
        cmd += ["--batch", str(batch)]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    for key, typ in (("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool),
                     ("scaling", str), ("dtype", str), ("data", str), ("config", dict),
                     ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), (key, d.get(key))
    assert d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["vs_baseline"] is None
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["unit"] == unit
    # the config names the workload's sizes exactly as the GPU arm's line does
    from attn_fwd_07_b300 import inputs
    spec = inputs.WORKLOADS[name]
    assert d["config"][cfg_key] == bench.workload_shape(spec.kind,
                                                        inputs.make(spec.name, batch), spec)
