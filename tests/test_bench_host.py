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
