"""Host-side checks of libbs.so (no GPU): exports, mesh builder vs the oracle."""

import os
import re
import subprocess
import types

import numpy as np
import pytest

import bsinputs as gen
import oracle
from conftest import ROOT, build_lib, oracle_ids


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
        bs.Mesh(2, 2, 1, flags=16)


def _expected_csr(ids, NG):
    order = np.argsort(ids, kind="stable")
    order = order[ids[order] >= 0]
    counts = np.bincount(ids[ids >= 0], minlength=NG)
    rs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return rs, order.astype(np.int32)


CASES = [("tiny", None), ("mid", None), ((2, 2, 0), None), ((3, 4, 7), None), ((1, 1, 3), None),
         ((5, 3, 3), 8), ((4, 2, 7), 100), ((6, 5, 3), 4096), ((3, 4, 15), None), ((4, 2, 8), 100),
         ((5, 5, 11), None), ((2, 7, 12), 8)]



@pytest.mark.parametrize("which,seg", CASES)
def test_mesh_builder_matches_oracle(bs, which, seg):
    if isinstance(which, str):
        cfg = gen.WORKLOADS[which]
    else:
        E, N, flags = which
        cfg = gen.MeshConfig("t", E, N, 0xABC + E, flags)
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags, seg_target=seg)
    assert m.validate() == bs.BS_OK
    assert (m.NL, m.NG, m.K) == (cfg.NL, cfg.NG, cfg.K)
    t = m.tables()
    ids = oracle_ids(cfg)
    assert np.array_equal(t["scatterIds"], ids)
    rs, li = _expected_csr(ids, cfg.NG)
    assert np.array_equal(t["rowStarts"], rs)
    assert np.array_equal(t["localIds"], li)
    assert m.nnz == int((ids >= 0).sum())
    masked_small = cfg.flags & gen.MASK_BOUNDARY and cfg.E < 2
    assert m.max_row == (8 if cfg.E >= 2 else (0 if masked_small else 1))
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


RANDOM_TABLES = [(5000, 1000, 0), (20000, 4000, 40), (3000, 100, 0), (1, 5, 0), (64, 64, 255),
                 (30000, 25000, 10)]


@pytest.mark.parametrize("NL,NG,masked", RANDOM_TABLES)
def test_mesh_from_ids_matches_numpy(bs, NL, NG, masked):
    """Tables of an arbitrary (unstructured) local-to-global map."""
    ids = gen.random_scatter_ids(NL + NG, 1, NL, NG, masked)
    m = bs.Mesh.from_ids(ids, NG)
    assert m.validate() == bs.BS_OK
    assert (m.NL, m.NG, m.E, m.N) == (NL, NG, 0, 0)
    t = m.tables()
    assert np.array_equal(t["scatterIds"], ids)
    rs, li = _expected_csr(ids, NG)
    assert np.array_equal(t["rowStarts"], rs) and np.array_equal(t["localIds"], li)
    assert m.nnz == int((ids >= 0).sum())
    lens = np.diff(rs)
    assert m.max_row == (int(lens.max()) if NG else 0)
    assert m.plan_info().valid == (m.max_row <= 32)


def test_mesh_from_ids_rejects_bad_tables(bs):
    with pytest.raises(bs.BSError) as e:
        bs.Mesh.from_ids(np.array([0, 5, 1], dtype=np.int32), 5)      # 5 >= NG
    assert e.value.status == bs.BS_EBOUNDS
    with pytest.raises(bs.BSError):
        bs.Mesh.from_ids(np.array([0, -2], dtype=np.int32), 3)        # below -1
    with pytest.raises(bs.BSError) as e:
        bs.Mesh.from_ids(np.zeros(5000, dtype=np.int32), 2)          # a row of 5000 > 4096
    assert e.value.status == bs.BS_EINVAL
    m = bs.Mesh.from_ids(np.zeros(40, dtype=np.int32), 3)             # 40 > 32: no plan
    assert m.validate() == bs.BS_OK and not m.plan_info().valid


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


# ------------------------------------------------- two-pass plan (host)

def _seq_row_sums(vals, starts, lens, strides):
    """Row sums from +0.0 in ascending order (vectorised over rows); entry k
    of a row sits at start + k * stride."""
    s = np.zeros(len(starts))
    for k in range(int(lens.max()) if len(lens) else 0):
        m = lens > k
        s[m] = s[m] + vals[starts[m] + k * strides[m]]
    return s


def simulate_plan_scatter(pt, pi, tabs, qG, NL):
    T, B, BL = pi.s_ntiles, pi.s_nbuckets, pi.s_bucket_len * pi.cluster
    rs, tr = tabs["rowStarts"], pt["s_tileRows"]
    run = pt["s_runStart"].reshape(T + 1, B)
    work = np.full(len(pt["s_src"]), np.nan)
    for t in range(T):
        r0, r1 = tr[t], tr[t + 1]
        off = np.concatenate([[0], np.cumsum(run[t + 1] - run[t])])
        assert off[-1] == rs[r1] - rs[r0]
        k = np.arange(off[-1])
        c = np.searchsorted(off, k, side="right") - 1
        src = pt["s_src"][rs[r0] + k].astype(np.int64)
        # bit 15 marks exactly the first slot of every non-empty run
        first = np.zeros(off[-1], bool)
        first[off[:-1][np.diff(off) > 0]] = True
        assert np.array_equal(src >= 0x8000, first)
        work[run[t][c] + (k - off[c])] = qG[r0:r1][src & 0x7FFF]
    qL = np.zeros(NL)
    for b in range(B):
        j0, j1 = run[0, b], run[T, b]
        qL[b * BL + pt["s_dst"][j0:j1].astype(np.int64)] = work[j0:j1]
    return qL


def simulate_plan_gather(pt, pi, tabs, qL, NG):
    U, C, TL, CS, MM = pi.g_ntiles, pi.g_nbuckets, pi.g_tile_len * pi.cluster, pi.cluster, pi.g_mmax
    rs, ts = tabs["rowStarts"], pt["g_tileSlot"]
    sub = pt["g_subRows"]
    assert len(sub) == CS * C + 1 and np.all(np.diff(sub) >= 0)
    sub_entries = rs[sub[1:]] - rs[sub[:-1]]
    assert sub_entries.max() <= pi.g_bucket_entries and np.diff(sub).max() <= pi.g_bucket_entries
    gs = pt["g_groupStart"].astype(np.int64).reshape(CS * C, MM + 1)
    rowpos = pt["g_rowPos"].astype(np.int64)
    run = pt["g_runStart"].reshape(U + 1, C)
    work = np.full(len(pt["g_src"]), np.nan)
    for u in range(U):
        off = np.concatenate([[0], np.cumsum(run[u + 1] - run[u])])
        assert off[-1] == ts[u + 1] - ts[u]
        k = np.arange(off[-1])
        c = np.searchsorted(off, k, side="right") - 1
        src = pt["g_src"][ts[u] + k].astype(np.int64)
        first = np.zeros(off[-1], bool)
        first[off[:-1][np.diff(off) > 0]] = True
        assert np.array_equal(src >= 0x8000, first)
        work[run[u][c] + (k - off[c])] = qL[u * TL:(u + 1) * TL][src & 0x7FFF]
    qG = np.zeros(NG)
    for c in range(C):
        E0, E1 = rs[sub[c * CS]], rs[sub[c * CS + CS]]
        assert run[0, c] == E0 and run[U, c] == E1
        vals = np.full(E1 - E0, np.nan)
        vals[pt["g_pos"][E0:E1].astype(np.int64)] = work[E0:E1]
        assert not np.any(np.isnan(vals))
        for j in range(CS):
            sb = c * CS + j
            r0, r1 = sub[sb], sub[sb + 1]
            lens = np.diff(rs[r0:r1 + 1])
            assert gs[sb, 0] == 0 and gs[sb, MM] == lens.sum()
            for m in range(1, MM + 1):
                nm = int((lens == m).sum())
                assert gs[sb, m] - gs[sb, m - 1] == m * nm
                # rows of length m: an m x nm column-major block, rows in
                # ascending order, entry k of a row nm slots after entry k-1
                pos = rowpos[r0:r1][lens == m]
                assert np.array_equal(pos, gs[sb, m - 1] + np.arange(nm))
            full = lens > 0
            assert np.all(rowpos[r0:r1][~full] == 0xFFFF)
            starts = rs[r0] - E0 + rowpos[r0:r1][full]
            lf = lens[full]
            strides = (gs[sb, lf] - gs[sb, lf - 1]) // lf
            out = np.zeros(r1 - r0)
            out[full] = _seq_row_sums(vals, starts, lf, strides)
            qG[r0:r1] = out
    return qG


PLAN_CASES = [("tiny", None), ("tiny", (100, 64, 200, 150, 1)), ("tiny", (100, 64, 200, 150, 2)),
              ("tiny", (100, 64, 200, 150, 4)), ("tiny", (7, 5, 9, 8, 1)), ("tiny", (7, 5, 9, 8, 4)),
              ("mid", None), ("mid", (16384, 24576, 16384, 22528, 2)),
              ((5, 3, 7), (300, 256, 500, 333, 2)), ((3, 4, 3), None), ((2, 2, 7), (4, 3, 5, 8, 4))]


@pytest.mark.parametrize("which,sizes", PLAN_CASES + [
    (("ids", 20000, 4000, 40), None), (("ids", 20000, 4000, 40), (300, 257, 500, 400, 1)),
    (("ids", 9000, 800, 0), (64, 100, 80, 90, 2)), (("ids", 30000, 25000, 10), None)])
def test_two_pass_plan_reproduces_oracle(bs, which, sizes):
    if isinstance(which, tuple) and which[0] == "ids":
        _, NL, NG, masked = which
        ids = gen.random_scatter_ids(NL + NG, 1, NL, NG, masked)
        m = bs.Mesh.from_ids(ids, NG)
        cfg = types.SimpleNamespace(NL=NL, NG=NG, seed=NL + NG)
    elif isinstance(which, str):
        cfg = gen.WORKLOADS[which]
        m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    else:
        E, N, flags = which
        cfg = gen.MeshConfig("t", E, N, 0x51 + E, flags)
        m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    if sizes is not None:
        assert m.plan(*sizes) == bs.BS_OK
    pi = m.plan_info()
    assert pi.valid
    assert max(pi.smem_s1, pi.smem_s2, pi.smem_g1, pi.smem_g2) <= 232448
    pt, tabs = m.plan_tables(), m.tables()
    ids = tabs["scatterIds"]
    qG = gen.uniform_pm1(cfg.seed, gen.TAG_U, cfg.NG)
    qL = gen.uniform_pm1(cfg.seed, gen.TAG_P, cfg.NL)
    got_s = simulate_plan_scatter(pt, pi, tabs, qG, cfg.NL)
    assert np.array_equal(got_s.view(np.uint64), oracle.scatter(ids, qG).view(np.uint64))
    got_g = simulate_plan_gather(pt, pi, tabs, qL, cfg.NG)
    assert np.array_equal(got_g.view(np.uint64), oracle.gather(ids, qL, cfg.NG).view(np.uint64))


def test_plan_rejects_bad_sizes_and_oversized_smem(bs):
    m = bs.Mesh(4, 3, 1)
    pi = m.plan_info()
    assert pi.valid and pi.cluster == 1 and pi.s_tile_rows == 24576
    assert m.plan(0, 10, 10, 10, 1) == bs.BS_EINVAL and not m.plan_info().valid
    assert m.plan(10, 70000, 10, 10, 1) == bs.BS_EINVAL
    assert m.plan(30000, 30000, 30000, 30000, 1) == bs.BS_EINVAL   # > 227 KB of shared memory
    assert m.plan(24576, 24576, 24576, 22528, 4) == bs.BS_EINVAL   # offsets beyond 15 / 16 bits
    assert m.plan(16385, 100, 100, 100, 2) == bs.BS_EINVAL         # tile offsets beyond 15 bits
    assert m.plan(100, 100, 16385, 100, 2) == bs.BS_EINVAL
    assert m.plan(100, 100, 100, 100, 3) == bs.BS_EINVAL           # cluster of 3
    assert m.plan(16384, 24576, 16384, 22528, 2) == bs.BS_OK and m.plan_info().valid


def test_fault_injection_on_the_host(bs, monkeypatch):
    """BS_FAULT fakes failures on the host, without a GPU."""
    monkeypatch.setenv("BS_FAULT", "alloc")
    with pytest.raises(bs.BSError) as e:
        bs.Context(0)
    assert e.value.status == bs.BS_ENOMEM
    monkeypatch.setenv("BS_FAULT", "launch,badtable")
    assert bs.Mesh(4, 3, 1).validate() == bs.BS_EBOUNDS
    ids = (np.arange(40, dtype=np.int32) % 7).astype(np.int32)
    assert bs.Mesh.from_ids(ids, 7).validate() == bs.BS_EBOUNDS
    monkeypatch.setenv("BS_FAULT", "")
    assert bs.Mesh(4, 3, 1).validate() == bs.BS_OK
    assert bs.Mesh.from_ids(ids, 7).validate() == bs.BS_OK
