import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")

# Planned gather/scatter on small meshes must exercise the two-pass kernels:
# contexts created during the tests keep the plan whatever the size (a test
# that wants the library default makes its own context).
os.environ.setdefault("BS_TUNE_ONEPASS", "0")


def build_lib():
    """Build libbs.so (if stale) without importing the package first."""
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_bs_libbuild", os.path.join(ROOT, "order_fem_cg_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # Test modules import the package at collection time, which maps
    # libbs.so into this process: rebuild a stale library before that, or
    # the whole session would run the previous build.
    build_lib()


def oracle_ids(cfg):
    """The oracle's local-to-global table of a mesh workload, honouring all
    of its flags (element order, global numbering, mask, orientations)."""
    import bsinputs as gen
    import oracle
    ep, npm = gen.mesh_perms(cfg)
    orient = gen.element_orientations(cfg) if cfg.flags & gen.ROTATE_ELEMS else None
    return oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm, bool(cfg.flags & gen.MASK_BOUNDARY),
                                  orient)


def read_golden(name):
    """Rows of a golden fixture, comments stripped, as lists of tokens."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden
