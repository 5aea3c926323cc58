"""The oracle's loops on every core (oracle/oracle_omp.c), the bench's
all-core CPU baseline: elementwise operations, scatter and gather bitwise
equal to the single-thread oracle; norm and dot (Dot2 per thread chunk,
chunks combined in order) equal to it within the accuracy of Dot2; the rows
of a table equal a sort by global id; the runner prints one sane JSON line."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bsinputs as gen
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(oracle.build_omp() is None, reason="no OpenMP C compiler")


def same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint64), np.asarray(b).view(np.uint64))


def test_elementwise_and_reductions_match_the_oracle():
    rng = np.random.default_rng(3)
    for n in (0, 1, 7, 1000, 1_000_003):
        x, y, z, w = (rng.standard_normal(n) * np.exp(rng.uniform(-20, 20, n)) for _ in range(4))
        assert same(oracle.omp_copy(x), oracle.copy(x))
        for beta in (1.0, -0.5):
            assert same(oracle.omp_axpy(0.37, x, beta, y), oracle.axpy(0.37, x, beta, y))
        a, b = oracle.omp_cg_update(0.61, x, y, z, w), oracle.cg_update(0.61, x, y, z, w)
        assert same(a[0], b[0]) and same(a[1], b[1])
        for got, ref in ((oracle.omp_dot(x, y), oracle.dot(x, y)), (oracle.omp_norm(x), oracle.norm(x)),
                         (a[2], b[2])):
            assert abs(got - ref) <= 1e-15 * max(abs(ref), 1e-300)


@pytest.mark.parametrize("masked", [0, 30])
def test_scatter_gather_and_rows_match_the_oracle(masked):
    NL, NG = 200_000, 70_000
    ids = gen.random_scatter_ids(NL + NG, 3, NL, NG, masked)
    starts, local = oracle.rows_of(ids, NG)
    keep = np.nonzero(ids >= 0)[0]
    ref = keep[np.argsort(ids[keep], kind="stable")]
    assert np.array_equal(local, ref)
    assert starts[0] == 0 and starts[-1] == keep.size
    assert np.array_equal(np.diff(starts), np.bincount(ids[keep], minlength=NG))
    qG = gen.uniform_pm1(5, 1, NG)
    qL = gen.uniform_pm1(5, 2, NL)
    assert same(oracle.omp_scatter(ids, qG), oracle.scatter(ids, qG))
    assert same(oracle.omp_gather((starts, local), qL, NG), oracle.gather(ids, qL, NG))


def test_box_mesh_gather_matches_the_oracle():
    cfg = gen.WORKLOADS["tiny"]
    ep, npm = gen.mesh_perms(cfg)
    ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm)
    qL = gen.uniform_pm1(cfg.seed, gen.TAG_U, cfg.NL)
    assert same(oracle.omp_gather(oracle.rows_of(ids, cfg.NG), qL, cfg.NG),
                oracle.gather(ids, qL, cfg.NG))


def test_runner_prints_one_json_line(tmp_path):
    cfg = gen.WORKLOADS["tiny"]
    ep, npm = gen.mesh_perms(cfg)
    path = tmp_path / "ids.npy"
    np.save(path, oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm))
    for extra in ([str(path)], []):
        res = subprocess.run([sys.executable, "-m", "oracle.allcores", "tiny", "0.2", *extra],
                             cwd=ROOT, capture_output=True, text=True, timeout=300)
        assert res.returncode == 0, res.stderr
        d = json.loads(res.stdout.strip().splitlines()[-1])
        assert d["workload"] == "tiny" and d["threads"] >= 1 and d["reps"] >= 1
        assert d["s_per_step"] > 0
        assert set(d["s_per_op"]) == {"copy", "axpy", "norm", "dot", "cg_update", "gather", "scatter",
                                      "cg_iteration"}
