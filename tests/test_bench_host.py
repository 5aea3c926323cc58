"""bench.py pieces that run without a GPU: the reference (oracle) arm."""

import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, check=True, cwd=ROOT).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] == 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["higher_is_better"] is True
    host = rec["cpu_baseline"]["host"]
    assert host["nproc"] >= 1 and host["model"]


def test_reference_arm_maps_no_library():
    """The reference arm runs the oracle alone: it never maps libbs.so (the
    byte counts it needs are loaded without importing the package)."""
    code = ("import sys, runpy; sys.argv = ['bench.py', '--impl', 'reference', '--config', 'tiny', "
            "'--steps', '1', '--warmup', '0']\n"
            "try:\n    runpy.run_path('bench.py', run_name='__main__')\nexcept SystemExit:\n    pass\n"
            "maps = open('/proc/self/maps').read()\n"
            "print('LIBBS' if 'libbs.so' in maps else 'NOLIB', 'ORACLE' if 'liboracle' in maps else '')\n"
            "print('PKG' if 'order_fem_cg_gb300' in sys.modules else 'NOPKG')")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True,
                         cwd=ROOT).stdout
    assert "NOLIB ORACLE" in out and "NOPKG" in out


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, env=env, cwd=ROOT)
    assert res.returncode == 0 and res.stdout.strip() == ""


def _ncu_csv(path, launches):
    """An ncu --csv log of (kernel, dram bytes) launches, in ncu's layout."""
    rows = ['"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
            '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
            '"Metric Value"']
    for i, (k, b) in enumerate(launches):
        for m, v in (("dram__bytes_read.sum", b * 0.75), ("dram__bytes_write.sum", b * 0.25),
                     ("gpu__time_duration.sum", 1000.0)):
            rows.append(f'"{i}","1","python","h","void <unnamed>::{k}<1>(<unnamed>::PlanArgs)",'
                        f'"1","7","(1024, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler '
                        f'metrics","{m}","byte","{v}"')
    with open(path, "w") as f:
        f.write("==PROF== Connected\n" + "\n".join(rows) + "\n")


def test_traffic_from_per_kernel_captures(tmp_path, monkeypatch):
    """bench.py --traffic-from: the i-th captured launch of a kernel is its
    i-th occurrence in one step; an operation's bytes are the sum over its
    kernels, scaled from the capture mesh by its moved-bytes model."""
    import bench
    pm = bench.bs_perf()
    g = str(tmp_path / "g.csv")
    _ncu_csv(g, [("gather_tile_kernel", 3e8), ("gather_tile_kernel", 1.0)])
    b = str(tmp_path / "b.csv")
    _ncu_csv(b, [("gather_bucket_tm_kernel", 2e8)])
    d = str(tmp_path / "d.csv")
    _ncu_csv(d, [("dot_kernel", 5e7), ("dot_kernel", 9e7)])
    out = str(tmp_path / "t.json")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", out)
    assert bench.traffic_from_csv([g, b, d], "probe", "stress") == 0
    doc = json.load(open(out))["kernels"]
    cw, tw = bench.gen.WORKLOADS["probe"], bench.gen.WORKLOADS["stress"]
    sg = pm.moved_bytes("gather", tw.NL, tw.NG, tw.NL) / pm.moved_bytes("gather", cw.NL, cw.NG, cw.NL)
    assert doc["gather"]["measured_bytes"] == 5e8
    assert abs(doc["gather"]["bytes_per_launch"] - 5e8 * sg) < 1
    assert doc["norm"]["measured_bytes"] == 5e7 and doc["dot"]["measured_bytes"] == 9e7
    assert abs(doc["norm"]["scale"] - tw.NL / cw.NL) < 1e-12
    assert "scatter" not in doc and "copy" not in doc   # not captured


def test_all_cores_leg_reports_a_figure_or_why_not():
    """cpu_baseline.all_cores: the oracle's loops on every core, run in a
    process of its own; a figure with its thread count and per-operation
    split, or -- without an OpenMP compiler -- an `unavailable` reason."""
    import bench
    import oracle
    cfg = bench.gen.WORKLOADS["tiny"]
    rec = bench.all_cores_baseline(cfg, 0.2)
    if oracle.build_omp() is None:
        assert "unavailable" in rec
        return
    assert rec["unit"] == "GB/s" and rec["value"] > 0 and rec["cores"] >= 1
    assert set(rec["per_op"]) == {"copy", "axpy", "norm", "dot", "cg_update", "gather", "scatter",
                                  "cg_iteration"}
    assert all(v["GB/s"] > 0 for v in rec["per_op"].values())
