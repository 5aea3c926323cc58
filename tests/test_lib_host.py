"""Host-side checks of libbs.so (no GPU): exports, mesh builder vs the oracle."""

import os
import re
import subprocess

import numpy as np
import pytest

import bsinputs as gen
import oracle
from conftest import ROOT, build_lib


@pytest.fixture(scope="module")
def bs():
    build_lib()
    import order_fem_cg_gb300 as bs
    return bs


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(bs_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(bs):
    decl = declared_functions()
    assert len(decl) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", bs.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(bs_\w+)$", out, flags=re.M))
    missing = [f for f in decl if f not in exported]
    assert not missing, missing
    assert sorted(bs.EXPORTS) == decl
    for f in decl:
        getattr(bs.lib, f)


def test_strerror_and_null_context(bs):
    assert bs.lib.bs_strerror(0) == b"ok"
    assert bs.lib.bs_strerror(bs.BS_EBOUNDS) == b"index table entry out of range"
    assert bs.lib.bs_copy(None, 0, None, None, None) == bs.BS_EINVAL
    assert bs.lib.bs_ctx_create(0, None) == bs.BS_EINVAL


def test_mesh_rejects_bad_arguments(bs):
    for E, N, seg in [(0, 3, 2048), (2, 0, 2048), (2, 2, 4), (2, 2, 5000)]:
        with pytest.raises(bs.BSError):
            bs.Mesh(E, N, 1, seg_target=seg)
    with pytest.raises(bs.BSError):
        bs.Mesh(2, 2, 1, flags=8)


def _expected_csr(ids, NG):
    order = np.argsort(ids, kind="stable")
    order = order[ids[order] >= 0]
    counts = np.bincount(ids[ids >= 0], minlength=NG)
    rs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return rs, order.astype(np.int32)


CASES = [("tiny", None), ("mid", None), ((2, 2, 0), None), ((3, 4, 7), None), ((1, 1, 3), None),
         ((5, 3, 3), 8), ((4, 2, 7), 100), ((6, 5, 3), 4096)]


@pytest.mark.parametrize("which,seg", CASES)
def test_mesh_builder_matches_oracle(bs, which, seg):
    if isinstance(which, str):
        cfg = gen.CONFIGS[which]
    else:
        E, N, flags = which
        cfg = gen.MeshConfig("t", E, N, 0xABC + E, flags)
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags, seg_target=seg)
    assert m.validate() == bs.BS_OK
    assert (m.NL, m.NG, m.K) == (cfg.NL, cfg.NG, cfg.K)
    t = m.tables()
    ep, npm = gen.mesh_perms(cfg)
    ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm, bool(cfg.flags & gen.MASK_BOUNDARY))
    assert np.array_equal(t["scatterIds"], ids)
    rs, li = _expected_csr(ids, cfg.NG)
    assert np.array_equal(t["rowStarts"], rs)
    assert np.array_equal(t["localIds"], li)
    assert m.nnz == int((ids >= 0).sum())
    assert m.max_row == (8 if cfg.E >= 2 else 1)
    bsx = t["blockStarts"]
    assert bsx[0] == 0 and bsx[-1] == cfg.NG and np.all(np.diff(bsx) > 0)
    target = seg or bs.GATHER_SEG_DEFAULT
    ent = rs[bsx[1:]] - rs[bsx[:-1]]
    rows = np.diff(bsx)
    assert np.all(ent <= target) and np.all(rows <= target)
    assert m.seg_max == max(int(ent.max()), int(rows.max()))
    # greedy: a segment ends only when the next row would overflow it
    nxt = rs[np.minimum(bsx[1:-1] + 1, cfg.NG)] - rs[bsx[1:-1]]
    assert np.all((ent[:-1] + nxt > target) | (rows[:-1] + 1 > target))


def test_masked_mesh_builder_matches_oracle(bs):
    cfg = gen.MeshConfig("m", 4, 3, 99, gen.SHUFFLE_ELEMS | gen.PERMUTE_GLOBAL | gen.MASK_BOUNDARY)
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    assert m.validate() == bs.BS_OK
    ep, npm = gen.mesh_perms(cfg)
    ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm, True)
    t = m.tables()
    assert np.array_equal(t["scatterIds"], ids)
    assert (ids < 0).sum() > 0 and m.nnz == (ids >= 0).sum()
    rs, li = _expected_csr(ids, cfg.NG)
    assert np.array_equal(t["rowStarts"], rs) and np.array_equal(t["localIds"], li)


def test_seeded_permutation_matches_generator(bs):
    """The library's internal SplitMix64 permutation equals the generator's."""
    cfg = gen.MeshConfig("p", 7, 1, 0xDEADBEEF)
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, gen.PERMUTE_GLOBAL)
    # degree 1, unshuffled elements: the local node (0,0,0) of slot s is the
    # lattice corner of element s, so scatterIds reveals nodePerm there.
    ids = m.tables()["scatterIds"].reshape(cfg.K, 8)
    npm = gen.permutation(cfg.seed, gen.TAG_NODE_PERM, cfg.NG)
    e = np.arange(cfg.K)
    ex, ey, ez = e % 7, (e // 7) % 7, e // 49
    M = 8
    assert np.array_equal(ids[:, 0], npm[ex + M * (ey + M * ez)])
