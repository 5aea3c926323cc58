"""GPU parity: the sm_103a kernels through the C ABI against the CPU oracle.

Tolerances: copy, AXPY, the fused update's x and r, scatter and gather are
bit-exact; norm, dot and the fused residual r.r are within 1e-12 relative
of the oracle's Dot2 value (the reductions sum in a different order), and
every reduction is bitwise reproducible run to run.
"""

import types

import numpy as np
import pytest

import bsinputs as gen
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from conftest import build_lib, oracle_ids  # noqa: E402

build_lib()
import order_fem_cg_gb300 as bs  # noqa: E402

DEV = torch.device("cuda", 0)
RTOL_RED = 1e-12

SIZES = [0, 1, 2, 3, 4, 5, 7, 31, 257, 1000, 4099, 65536 + 3, 1000003]
OFFSETS = [(0, 0), (1, 1), (2, 2), (3, 3), (1, 0), (0, 2), (2, 3)]


def dev(a, offset=0):
    """Device copy of a at element offset `offset` inside a larger buffer (misaligned views)."""
    buf = torch.empty(a.size + offset + 1, dtype=torch.float64, device=DEV)
    v = buf[offset:offset + a.size]
    v.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return v


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits_equal(a, b):
    return np.array_equal(np.asarray(a).view(np.uint64), np.asarray(b).view(np.uint64))


def rel_close(got, ref, rtol=RTOL_RED):
    return abs(got - ref) <= rtol * abs(ref) or (ref == 0.0 and got == 0.0)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("off", OFFSETS)
def test_copy(n, off):
    x = gen.uniform_pm1(1, 7, n)
    xd, yd = dev(x, off[0]), dev(np.zeros(n), off[1])
    bs.bs_copy(xd, yd)
    assert bits_equal(host(yd), oracle.copy(x))


@pytest.mark.parametrize("beta", [1.0, -0.5, 0.3])
@pytest.mark.parametrize("n", [0, 1, 5, 1000, 65536 + 3, 1000003])
@pytest.mark.parametrize("off", [(0, 0), (3, 3), (1, 2)])
def test_axpy(beta, n, off):
    x = gen.uniform_pm1(2, 7, n)
    y = gen.uniform_pm1(2, 9, n)
    xd, yd = dev(x, off[0]), dev(y, off[1])
    bs.bs_axpy(0.37, xd, beta, yd)
    assert bits_equal(host(yd), oracle.axpy(0.37, x, beta, y))


def test_axpy_aliased():
    x = gen.uniform_pm1(3, 7, 100003)
    xd = dev(x, 1)
    bs.bs_axpy(0.37, xd, 1.0, xd)
    assert bits_equal(host(xd), oracle.axpy(0.37, x, 1.0, x))


@pytest.mark.parametrize("n", SIZES + [1 << 22])
@pytest.mark.parametrize("off", [(0, 0), (1, 1), (3, 3), (1, 2)])
def test_norm_and_dot(n, off):
    x = gen.uniform_pm1(4, 7, n)
    y = gen.uniform_pm1(4, 9, n)
    xd, yd = dev(x, off[0]), dev(y, off[1])
    nr = host(bs.bs_norm(xd))[0]
    dt = host(bs.bs_dot(xd, yd))[0]
    assert rel_close(nr, oracle.norm(x))
    assert rel_close(dt, oracle.dot(x, y))
    # run to run: bitwise identical
    assert bits_equal(host(bs.bs_norm(xd)), [nr])
    assert bits_equal(host(bs.bs_dot(xd, yd)), [dt])
    if n == 0:
        assert not np.signbit(nr) and not np.signbit(dt)


def test_norm_closed_forms():
    n = 1000003
    assert host(bs.bs_norm(dev(np.full(n, 0.5))))[0] == n / 4
    i = np.arange(n, dtype=np.float64)
    exact = (n - 1) * n * (2 * n - 1) // 6
    assert abs(host(bs.bs_norm(dev(i)))[0] - exact) <= 1e-12 * exact
    assert host(bs.bs_dot(dev(i), dev(np.ones(n))))[0] == n * (n - 1) // 2


@pytest.mark.parametrize("log2n", [10, 17, 27])
def test_sweep_points(log2n):
    x, y, alpha = gen.sweep_vectors(log2n)
    xd, yd = dev(x), dev(y)
    assert rel_close(host(bs.bs_norm(xd))[0], oracle.norm(x))
    assert rel_close(host(bs.bs_dot(xd, yd))[0], oracle.dot(x, y))
    bs.bs_axpy(alpha, xd, 1.0, yd)
    assert bits_equal(host(yd), oracle.axpy(alpha, x, 1.0, y))
    zd = dev(np.zeros(x.size))
    bs.bs_copy(xd, zd)
    assert bits_equal(host(zd), x)


@pytest.mark.parametrize("n", [0, 1, 3, 6, 1000, 65536 + 3, 1000003])
@pytest.mark.parametrize("off", [(0, 0, 0, 0), (1, 1, 1, 1), (0, 1, 2, 3)])
def test_cg_update(n, off):
    p, Ap, x, r = (gen.uniform_pm1(5, t, n) for t in (gen.TAG_P, gen.TAG_AP, gen.TAG_X, gen.TAG_R))
    alpha = 0.37
    pd, Apd, xd, rd = dev(p, off[0]), dev(Ap, off[1]), dev(x, off[2]), dev(r, off[3])
    rr = host(bs.bs_cg_update(pd, Apd, xd, rd, alpha=alpha))[0]
    xo, ro, rro = oracle.cg_update(alpha, p, Ap, x, r)
    assert bits_equal(host(xd), xo) and bits_equal(host(rd), ro)
    assert rel_close(rr, rro)
    assert rel_close(rr, oracle.norm(host(rd)))


def test_cg_update_device_alpha_and_no_reduction():
    n = 300007
    p, Ap, x, r = (gen.uniform_pm1(6, t, n) for t in (4, 5, 7, 6))
    num = torch.tensor([0.8], dtype=torch.float64, device=DEV)
    den = torch.tensor([3.0], dtype=torch.float64, device=DEV)
    alpha = 0.8 / 3.0
    pd, Apd, xd, rd = dev(p), dev(Ap), dev(x), dev(r)
    rr = host(bs.bs_cg_update(pd, Apd, xd, rd, alpha_num=num, alpha_den=den))[0]
    xo, ro, rro = oracle.cg_update(alpha, p, Ap, x, r)
    assert bits_equal(host(xd), xo) and bits_equal(host(rd), ro) and rel_close(rr, rro)
    pd, Apd, xd, rd = dev(p), dev(Ap), dev(x), dev(r)
    assert bs.bs_cg_update(pd, Apd, xd, rd, alpha=alpha, reduce=False) is None
    assert bits_equal(host(xd), xo) and bits_equal(host(rd), ro)


def test_reductions_bitwise_reproducible_large():
    n = (1 << 25) + 12345
    x = gen.normal(7, 3, n)
    xd = dev(x, 1)
    vals = {host(bs.bs_norm(xd)).view(np.uint64)[0] for _ in range(5)}
    assert len(vals) == 1


# ------------------------------------------------------------- meshes

def mesh_case(cfg, seg=None, planned=False, sizes=None):
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags, seg_target=seg)
    assert m.validate() == bs.BS_OK
    if sizes is not None:
        assert m.plan(*sizes) == bs.BS_OK
    ids = m.tables()["scatterIds"]
    ids_o = oracle_ids(cfg)
    assert np.array_equal(ids, ids_o)
    t = m.to_device(0, planned=planned)
    assert (t.plan is not None) == planned
    return m, t, ids_o


MESHES = [
    (gen.WORKLOADS["tiny"], None),
    (gen.WORKLOADS["tiny"], 8),
    (gen.WORKLOADS["tiny"], 1000),
    (gen.WORKLOADS["tiny"], 4096),
    (gen.MeshConfig("masked", 6, 4, 17, 7), None),
    (gen.MeshConfig("plain", 5, 2, 3, 0), 3000),
    (gen.MeshConfig("one", 1, 1, 5, 3), None),
    (gen.MeshConfig("onemask", 1, 3, 5, 7), 8),
    (gen.MeshConfig("rot", 5, 3, 31, 11), None),
    (gen.MeshConfig("rotmask", 4, 5, 32, 15), 1000),
    (gen.WORKLOADS["mid"], None),
]


PLANNED = [
    (gen.WORKLOADS["tiny"], None),
    (gen.WORKLOADS["tiny"], (100, 64, 200, 150, 1)),
    (gen.WORKLOADS["tiny"], (100, 64, 200, 150, 2)),
    (gen.WORKLOADS["tiny"], (100, 64, 200, 150, 4)),
    (gen.WORKLOADS["tiny"], (7, 5, 9, 8, 2)),
    (gen.WORKLOADS["tiny"], (7, 5, 9, 8, 4)),
    (gen.MeshConfig("masked", 6, 4, 17, 7), (500, 333, 700, 600, 2)),
    (gen.MeshConfig("masked4", 6, 4, 17, 7), (500, 333, 700, 600, 4)),
    (gen.MeshConfig("one", 1, 1, 5, 3), None),
    (gen.MeshConfig("onemask", 1, 3, 5, 7), (3, 5, 7, 9, 2)),
    (gen.MeshConfig("rot", 5, 3, 31, 11), None),
    (gen.MeshConfig("rotmask", 4, 5, 32, 15), (700, 500, 900, 800, 1)),
    (gen.MeshConfig("midrotmask", 20, 7, 33, 15), None),
    (gen.WORKLOADS["mid"], None),
    (gen.WORKLOADS["mid"], (16384, 24576, 16384, 22528, 2)),
    (gen.WORKLOADS["large"], None),
]


@pytest.mark.parametrize("cfg,seg", MESHES, ids=lambda v: getattr(v, "name", str(v)))
def test_scatter_gather(cfg, seg):
    check_scatter_gather(cfg, *mesh_case(cfg, seg))


@pytest.mark.parametrize("cfg,sizes", PLANNED, ids=lambda v: getattr(v, "name", str(v)))
def test_scatter_gather_two_pass(cfg, sizes):
    check_scatter_gather(cfg, *mesh_case(cfg, planned=True, sizes=sizes))


def check_scatter_gather(cfg, m, t, ids):
    qG = gen.uniform_pm1(cfg.seed, gen.TAG_U, cfg.NG)
    qL = gen.uniform_pm1(cfg.seed, gen.TAG_P, cfg.NL)
    qLd = dev(np.zeros(cfg.NL))
    bs.bs_scatter(t, dev(qG), qLd)
    assert bits_equal(host(qLd), oracle.scatter(ids, qG))
    qGd = dev(np.full(cfg.NG, np.nan))
    bs.bs_gather(t, dev(qL), qGd)
    assert bits_equal(host(qGd), oracle.gather(ids, qL, cfg.NG))
    assert bs.default_context().device_status() == bs.BS_OK


@pytest.mark.parametrize("idx_off,work_off", [(0, 0), (1, 0), (2, 0), (3, 1), (0, 1), (2, 3)])
def test_two_pass_with_shifted_plan_tables(idx_off, work_off):
    """Pass 2 reads its work entries four, two or one at a time depending on
    how the 16-bit position tables and the work array line up; shifting them
    (16-bit and 8-byte steps) runs every one of those paths, on a masked mesh
    (zeroed buckets) and its unmasked twin, for scatter, gather and the fused
    diagonal operator."""
    for flags in (7, 3):
        cfg = gen.MeshConfig("shift", 6, 4, 23, flags)
        m, t, ids = mesh_case(cfg, planned=True, sizes=(300, 500, 500, 400, 1))
        keep = []
        for name in ("s_dst", "g_pos"):
            src = t.plan[name]
            buf = torch.zeros(src.numel() + 4, dtype=torch.int16, device=DEV)
            buf[idx_off:idx_off + src.numel()] = src
            keep.append(buf)
            setattr(t.plan_struct, name, buf.data_ptr() + 2 * idx_off)
        work = torch.empty(2 * m.nnz + 4, dtype=torch.float64, device=DEV)
        keep.append(work)
        t.plan_struct.work = work.data_ptr() + 8 * work_off
        check_scatter_gather(cfg, m, t, ids)
        dL = gen.uniform_range(cfg.seed, 1, cfg.NL, 0.5, 1.5)
        x = gen.uniform_pm1(cfg.seed, 2, cfg.NG)
        y = torch.empty(cfg.NG, dtype=torch.float64, device=DEV)
        bs.bs_apply_diag(t, dev(x), dev(dL), y)
        assert bits_equal(host(y), oracle.apply_diag(ids, dL, x))
        assert bs.default_context().device_status() == bs.BS_OK
        del keep


@pytest.mark.parametrize("NL,NG,masked,planned", [
    (20000, 4000, 40, False), (20000, 4000, 40, True), (300000, 120000, 0, True),
    (3000, 100, 0, False), (3000, 100, 0, True), (2000000, 400000, 25, True),
    (20000, 600, 0, False)])
def test_scatter_gather_random_tables(NL, NG, masked, planned):
    """Any local-to-global map (bs_mesh_from_ids): rows of Poisson length,
    masked locals, empty rows; rows longer than 32 (NL/NG = 33) leave the
    plan invalid and use the one-pass kernels."""
    ids = gen.random_scatter_ids(NL + NG, 3, NL, NG, masked)
    m = bs.Mesh.from_ids(ids, NG)
    assert m.validate() == bs.BS_OK
    t = m.to_device(0, planned=planned and m.plan_info().valid)
    cfg = types.SimpleNamespace(NL=NL, NG=NG, seed=NL)
    check_scatter_gather(cfg, m, t, ids)
    if planned and m.plan_info().valid:
        dL = gen.uniform_range(7, 1, NL, 0.5, 1.5)
        x = gen.uniform_pm1(7, 2, NG)
        y = torch.empty(NG, dtype=torch.float64, device=DEV)
        bs.bs_apply_diag(t, dev(x), dev(dL), y)
        assert bits_equal(host(y), oracle.apply_diag(ids, dL, x))


@pytest.mark.parametrize("planned", [False, True])
def test_scatter_gather_unaligned_views(planned):
    cfg = gen.WORKLOADS["tiny"]
    m, t, ids = mesh_case(cfg, planned=planned)
    qG = gen.uniform_pm1(1, 1, cfg.NG)
    qLd = dev(np.zeros(cfg.NL), 1)            # 8-byte aligned only
    bs.bs_scatter(t, dev(qG, 3), qLd)
    assert bits_equal(host(qLd), oracle.scatter(ids, qG))
    qL = gen.uniform_pm1(1, 2, cfg.NL)
    qGd = dev(np.zeros(cfg.NG), 1)
    bs.bs_gather(t, dev(qL, 3), qGd)
    assert bits_equal(host(qGd), oracle.gather(ids, qL, cfg.NG))


@pytest.mark.parametrize("planned", [False, True])
def test_gather_sum_order_probe(planned):
    """Rows whose sum depends on order: 1.0 at the smallest local id, 2^-53 elsewhere."""
    cfg = gen.WORKLOADS["tiny"]
    m, t, ids = mesh_case(cfg, planned=planned, sizes=(50, 40, 60, 64, 2) if planned else None)
    tabs = m.tables()
    rs, li = tabs["rowStarts"], tabs["localIds"]
    for first in (True, False):
        qL = np.full(cfg.NL, 2.0 ** -53)
        pick = rs[:-1] if first else rs[1:] - 1
        qL[li[pick]] = 1.0
        qGd = dev(np.zeros(cfg.NG))
        bs.bs_gather(t, dev(qL), qGd)
        assert bits_equal(host(qGd), oracle.gather(ids, qL, cfg.NG))


@pytest.mark.parametrize("planned", [False, True])
def test_gather_of_ones_and_identities(planned):
    cfg = gen.WORKLOADS["mid"]
    m, t, ids = mesh_case(cfg, planned=planned)
    mult = dev(np.zeros(cfg.NG))
    bs.bs_gather(t, dev(np.ones(cfg.NL)), mult)
    mh = host(mult)
    a, b = cfg.E - 1, cfg.E * (cfg.N - 1) + 2
    vals, counts = np.unique(mh, return_counts=True)
    assert dict(zip(vals.astype(int).tolist(), counts.tolist())) == {
        1: b ** 3, 2: 3 * a * b * b, 4: 3 * a * a * b, 8: a ** 3}
    u = gen.integers_dyadic(cfg.seed, 3, cfg.NG)
    qL = dev(np.zeros(cfg.NL))
    bs.bs_scatter(t, dev(u), qL)
    back = dev(np.zeros(cfg.NG))
    bs.bs_gather(t, qL, back)
    assert np.array_equal(host(back), mh * u)


def test_out_of_range_entry_is_flagged_not_dereferenced():
    cfg = gen.WORKLOADS["tiny"]
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    tabs = m.tables()
    bad_ids = tabs["scatterIds"].copy()
    bad_ids[123] = cfg.NG + 5               # beyond q_G: the kernel must skip it
    bad_local = tabs["localIds"].copy()
    bad_local[77] = cfg.NL + 1000           # beyond q_L
    tabs_bad = dict(tabs, scatterIds=bad_ids, localIds=bad_local)
    t = bs.DeviceTables.from_host(tabs_bad, m.info, 0)
    ctx = bs.default_context()
    assert ctx.device_status() == bs.BS_OK
    qG = gen.uniform_pm1(1, 1, cfg.NG)
    qLd = dev(np.zeros(cfg.NL))
    bs.bs_scatter(t, dev(qG), qLd)
    assert ctx.device_status() == bs.BS_EBOUNDS
    got = host(qLd)
    assert got[123] == 0.0
    good = np.ones(cfg.NL, bool)
    good[123] = False
    assert bits_equal(got[good], oracle.scatter(tabs["scatterIds"], qG)[good])
    qGd = dev(np.zeros(cfg.NG))
    bs.bs_gather(t, dev(gen.uniform_pm1(1, 2, cfg.NL)), qGd)
    assert ctx.device_status() == bs.BS_EBOUNDS
    assert ctx.device_status() == bs.BS_OK   # the flag was cleared by the read


@pytest.mark.parametrize("cluster", [1, 2])
def test_bad_plan_entry_is_flagged_not_dereferenced(cluster):
    cfg = gen.WORKLOADS["tiny"]
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    assert m.plan(100, 64, 200, 150, cluster) == bs.BS_OK
    pt, pi = m.plan_tables(), m.plan_info()
    for key, bad in (("s_dst", 65535), ("s_src", 65535), ("g_src", 65535), ("g_pos", 65535),
                     ("s_src", 0x7FFF), ("g_src", 0x7FFF)):
        corrupt = dict(pt)
        corrupt[key] = pt[key].copy()
        corrupt[key][17] = bad
        t = bs.DeviceTables.from_host(m.tables(), m.info, 0, (corrupt, pi))
        ctx = bs.default_context()
        assert ctx.device_status() == bs.BS_OK
        qLd, qGd = dev(np.zeros(cfg.NL)), dev(np.zeros(cfg.NG))
        bs.bs_scatter(t, dev(gen.uniform_pm1(1, 1, cfg.NG)), qLd)
        bs.bs_gather(t, dev(gen.uniform_pm1(1, 2, cfg.NL)), qGd)
        assert ctx.device_status() == bs.BS_EBOUNDS, key


def test_invalid_arguments_rejected():
    x = dev(np.zeros(10))
    with pytest.raises(ValueError):
        bs.bs_copy(x, x[:9])
    with pytest.raises(bs.BSError):
        bs.bs_copy(x[0:6], x[4:10])            # partial overlap
    cfg = gen.WORKLOADS["tiny"]
    m, t, ids = mesh_case(cfg)
    buf = torch.zeros(cfg.NL, dtype=torch.float64, device=DEV)
    with pytest.raises(bs.BSError):
        bs.bs_gather(t, buf, buf[:cfg.NG])     # qL and qG overlap
    p = dev(np.zeros(100))
    with pytest.raises(bs.BSError):
        bs.bs_cg_update(p, p, p, p, alpha=1.0)


# ---------------------------------------------------------- CG sequence

@pytest.mark.parametrize("name,planned", [("tiny", False), ("mid", False), ("tiny", True),
                                          ("mid", True)])
def test_cg_iteration_sequence(name, planned):
    cfg = gen.WORKLOADS[name]
    m, t, ids = mesh_case(cfg, planned=planned)
    NG = cfg.NG
    pG = gen.uniform_pm1(cfg.seed, gen.TAG_P, NG)
    xG = gen.uniform_pm1(cfg.seed, gen.TAG_X, NG)
    rG = gen.uniform_pm1(cfg.seed, gen.TAG_R, NG)
    rr = oracle.norm(rG)
    ref = oracle.cg_sequence(ids, pG, xG, rG, rr)
    pGd, xGd, rGd = dev(pG), dev(xG), dev(rG)
    pLd, ApGd = dev(np.zeros(cfg.NL)), dev(np.zeros(NG))
    sc = {k: torch.zeros(1, dtype=torch.float64, device=DEV) for k in ("pAp", "rr_new", "rnorm")}
    rrd = torch.tensor([rr], dtype=torch.float64, device=DEV)
    bs.bs_cg_iteration(t, pGd, pLd, ApGd, xGd, rGd, rrd, sc["pAp"], sc["rr_new"], sc["rnorm"])
    assert bits_equal(host(pLd), ref["pL"]) and bits_equal(host(ApGd), ref["ApG"])
    pAp = host(sc["pAp"])[0]
    assert rel_close(pAp, ref["pAp"])
    alpha = rr / pAp
    # x, r depend on alpha = rr / pAp, whose last bits follow the reduction
    # order: |dx| <= |d alpha| |p| + 1 ulp, |d alpha| <= 2e-12 |alpha|.
    da = 2e-12 * abs(ref["alpha"])
    for got, exp, v in ((host(xGd), ref["x"], pG), (host(rGd), ref["r"], host(ApGd))):
        assert np.all(np.abs(got - exp) <= da * np.abs(v) + np.spacing(np.abs(exp)))
    assert rel_close(host(sc["rr_new"])[0], ref["rr_new"], 1e-11)
    assert rel_close(host(sc["rnorm"])[0], oracle.norm(host(rGd)))
    assert bits_equal(host(sc["rnorm"]), host(sc["rr_new"])) or rel_close(
        host(sc["rnorm"])[0], host(sc["rr_new"])[0])
    assert abs(alpha - ref["alpha"]) <= da


def wide_range_vector(n, seed):
    """Mantissas U(1,2) times 2^k, k in [-70, 70], random signs, with zeros and subnormals."""
    m = 1.0 + (gen.uniform_pm1(seed, 1, n) + 1.0) / 2.0
    k = np.floor((gen.uniform_pm1(seed, 2, n) + 1.0) * 70.5 - 70.0).astype(int)
    x = np.ldexp(m, k) * np.sign(gen.uniform_pm1(seed, 3, n))
    x[::97] = 0.0
    x[5::211] = -0.0
    x[7::503] = 5e-324 * np.arange(1, x[7::503].size + 1)
    x[11::1009] = 2.0 ** 41      # exactly at the fast-range edge
    x[13::1013] = 2.0 ** -40
    return x


@pytest.mark.parametrize("n", [1, 8, 1000, 1000003])
def test_norm_wide_exponent_range(n):
    x = wide_range_vector(n, 17)
    got = host(bs.bs_norm(dev(x, 1)))[0]
    assert rel_close(got, oracle.norm(x))
    # each binade alone (sums dominated by one magnitude)
    for k in (-45, -40, -39, 0, 40, 41, 60):
        y = np.ldexp(1.0 + (gen.uniform_pm1(k + 100, 4, 4099) + 1.0) / 2.0, k)
        assert rel_close(host(bs.bs_norm(dev(y)))[0], oracle.norm(y))


def test_fused_residual_wide_exponent_range():
    n = 300007
    r = wide_range_vector(n, 23)
    p, Ap, x = (gen.uniform_pm1(9, t, n) for t in (4, 5, 7))
    pd, Apd, xd, rd = dev(p), dev(Ap), dev(x), dev(r)
    rr = host(bs.bs_cg_update(pd, Apd, xd, rd, alpha=1e-30))[0]
    xo, ro, rro = oracle.cg_update(1e-30, p, Ap, x, r)
    assert bits_equal(host(rd), ro) and rel_close(rr, rro)


def _all_low_bits(x):
    """x with the 29 low fraction bits set: the 6 bits the float-float split
    drops, and the 23 it keeps in xl, are all ones."""
    b = np.abs(x).view(np.uint64) | np.uint64((1 << 29) - 1)
    return b.view(np.float64)


def worst_case_vectors(n):
    """Inputs that push the float-float sum of squares to its error bound:
    one sign, every value with its low fraction bits all ones (the dropped
    bits are maximal, so every square is under-estimated the same way), and
    8-element chunks built so that each float addition into s rounds with a
    large error: one dominant term then seven terms 2^-12 smaller in value
    (2^-24 in square, half an ulp of s), the same pattern reversed, and all
    terms equal to the largest double below 2."""
    top = np.nextafter(2.0, 0.0)
    equal = np.full(n, top)
    pat = np.empty(8)
    pat[0] = top
    pat[1:] = np.ldexp(top, -12)
    lead = np.tile(pat, n // 8 + 1)[:n]
    trail = np.tile(pat[::-1], n // 8 + 1)[:n]
    rnd = _all_low_bits(0.5 + 0.5 * (gen.uniform_pm1(71, 1, n) + 1.0) / 2.0)
    return {"equal": equal, "lead": lead, "trail": trail, "random_low_bits": rnd}


def test_norm_worst_case_at_2_27():
    """n = 2^27 (the sweep's largest size): every worst-case pattern within
    1e-12 of the oracle's Dot2 sum (the derived bound is 5e-13)."""
    n = 1 << 27
    for name, x in worst_case_vectors(n).items():
        xd = dev(x)
        got = host(bs.bs_norm(xd))[0]
        ref = oracle.norm(x)
        assert abs(got - ref) <= 1e-12 * ref, (name, got, ref, (got - ref) / ref)
        del xd
        torch.cuda.empty_cache()


def test_fused_residual_worst_case_at_2_27():
    """BS5's r.r uses the same accumulator: alpha = 0 keeps r bit for bit, so
    r.r is the sum of squares of the worst-case patterns."""
    n = 1 << 27
    pats = worst_case_vectors(n)
    p = torch.zeros(n, dtype=torch.float64, device=DEV)
    Ap = torch.zeros(n, dtype=torch.float64, device=DEV)
    x = torch.zeros(n, dtype=torch.float64, device=DEV)
    for name in ("equal", "lead", "random_low_bits"):
        r = dev(pats[name])
        rr = host(bs.bs_cg_update(p, Ap, x, r, alpha=0.0))[0]
        ref = oracle.norm(pats[name])
        assert abs(rr - ref) <= 1e-12 * ref, (name, rr, ref, (rr - ref) / ref)
        del r
        torch.cuda.empty_cache()


def test_norm_non_finite():
    x = gen.uniform_pm1(3, 3, 5000)
    x[1234] = np.inf
    assert host(bs.bs_norm(dev(x)))[0] == np.inf
    x[17] = np.nan
    assert np.isnan(host(bs.bs_norm(dev(x)))[0])


# ------------------------------------------- diagonal local operator (fused)

FUSED = [
    (gen.WORKLOADS["tiny"], None),
    (gen.WORKLOADS["tiny"], (100, 64, 64, 150, 1)),
    (gen.WORKLOADS["tiny"], (7, 9, 9, 8, 1)),
    (gen.MeshConfig("masked", 6, 4, 17, 7), (500, 333, 333, 600, 1)),
    (gen.MeshConfig("one", 1, 1, 5, 3), None),
    (gen.WORKLOADS["mid"], None),
    (gen.WORKLOADS["large"], None),
]


@pytest.mark.parametrize("cfg,sizes", FUSED, ids=lambda v: getattr(v, "name", str(v)))
def test_apply_diag(cfg, sizes):
    m, t, ids = mesh_case(cfg, planned=True, sizes=sizes)
    x = gen.uniform_pm1(cfg.seed, gen.TAG_X, cfg.NG)
    for d in (gen.mass_diagonal(cfg.E, cfg.N), 1.0 + 0.5 * gen.uniform_pm1(cfg.seed, 21, cfg.NL),
              np.ones(cfg.NL)):
        yd = dev(np.full(cfg.NG, np.nan))
        bs.bs_apply_diag(t, dev(x), dev(d), yd)
        assert bits_equal(host(yd), oracle.apply_diag(ids, d, x))
    assert bs.default_context().device_status() == bs.BS_OK


def adversarial_local_values(m, seed):
    """q_L values whose row sums exercise every corner of a binary64 addition:
    exponents over the whole range (subnormals included), signed zeros,
    values near the largest double (sums that overflow to infinity), a few
    +inf, rows whose entries cancel exactly or in all but their last bits, and
    rows that add half an ulp to an even or an odd significand (rounding
    ties)."""
    rng = np.random.default_rng(seed)
    NL = m.info.NL
    sign = np.where(rng.random(NL) < 0.5, -1.0, 1.0)
    mant = 1.0 + rng.random(NL)
    x = sign * np.ldexp(mant, rng.integers(-40, 41, NL))
    kind = rng.integers(0, 16, NL)
    x[kind == 0] = (sign * np.ldexp(mant, rng.integers(-1080, 1024, NL)))[kind == 0]
    x[kind == 1] = (sign * 0.0)[kind == 1]
    x[kind == 2] = np.ldexp(mant, 1023)[kind == 2]  # positive: sums overflow to +inf only (no inf - inf)
    x[(kind == 3) & (rng.random(NL) < 0.01)] = np.inf
    tabs = m.tables()
    rs, li = tabs["rowStarts"].astype(np.int64), tabs["localIds"].astype(np.int64)
    rows = np.nonzero(np.diff(rs) >= 2)[0]
    pick = rng.permutation(rows)
    n4 = len(pick) // 4
    a, b = li[rs[pick]], li[rs[pick] + 1]
    base = x[a]
    finite = np.isfinite(base) & (base != 0.0) & (np.abs(base) < 2.0 ** 1000)
    # exact cancellation, then cancellation in all but the last bits
    x[b[:n4]] = np.where(finite[:n4], -base[:n4], x[b[:n4]])
    flip = np.frombuffer(np.ascontiguousarray(base[n4:2 * n4]).tobytes(), dtype=np.uint64) ^ \
        rng.integers(1, 1 << 20, n4, dtype=np.uint64)
    near = -np.frombuffer(flip.tobytes(), dtype=np.float64)
    x[b[n4:2 * n4]] = np.where(finite[n4:2 * n4], near, x[b[n4:2 * n4]])
    # ties: 2^k (even significand) or 2^k (1 + 2^-52) (odd) plus 2^(k-53)
    k = rng.integers(-500, 500, len(pick) - 2 * n4)
    odd = rng.random(len(k)) < 0.5
    x[a[2 * n4:]] = np.ldexp(np.where(odd, 1.0 + 2.0 ** -52, 1.0), k)
    x[b[2 * n4:]] = np.ldexp(1.0, k - 53) * np.where(rng.random(len(k)) < 0.5, -1.0, 1.0)
    return x


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_gather_adversarial_values(name):
    """Row sums of adversarial values (see adversarial_local_values) through
    the two-pass gather and the one-pass gather, bit for bit against the
    oracle's ascending binary64 sums."""
    cfg = gen.WORKLOADS[name]
    for planned in (True, False):
        m, t, ids = mesh_case(cfg, planned=planned)
        for seed in (1, 2):
            qL = adversarial_local_values(m, seed + 10 * cfg.seed)
            out = dev(np.full(cfg.NG, np.nan))
            bs.bs_gather(t, dev(qL), out)
            assert bits_equal(host(out), oracle.gather(ids, qL, cfg.NG))
    assert bs.default_context().device_status() == bs.BS_OK


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_gather_pass2_without_tmem_buffer(name, monkeypatch):
    """Gather pass 2 has two kernels: by default the persistent one that
    stages the next bucket in tensor memory, and the one-bucket-per-block
    kernel (BS_TUNE_TMEM=0 at context creation).  Both are bit-exact to the
    oracle; this keeps the second one covered."""
    cfg = gen.WORKLOADS[name]
    m, t, ids = mesh_case(cfg, planned=True)
    monkeypatch.setenv("BS_TUNE_TMEM", "0")
    ctx = bs.Context()
    monkeypatch.delenv("BS_TUNE_TMEM")
    qL = gen.uniform_pm1(cfg.seed, gen.TAG_U, cfg.NL)
    ref = oracle.gather(ids, qL, cfg.NG)
    for c in (ctx, None):
        out = dev(np.full(cfg.NG, np.nan))
        bs.bs_gather(t, dev(qL), out, ctx=c)
        assert bits_equal(host(out), ref)
    x = gen.uniform_pm1(cfg.seed, gen.TAG_X, cfg.NG)
    d = gen.mass_diagonal(cfg.E, cfg.N)
    yd = dev(np.full(cfg.NG, np.nan))
    bs.bs_apply_diag(t, dev(x), dev(d), yd, ctx=ctx)
    assert bits_equal(host(yd), oracle.apply_diag(ids, d, x))
    assert ctx.device_status() == bs.BS_OK
    ctx.close()


def test_apply_diag_rejects_unfusable_plans():
    cfg = gen.WORKLOADS["tiny"]
    x, d = dev(np.ones(cfg.NG)), dev(np.ones(cfg.NL))
    for sizes in ((100, 64, 128, 150, 1), (100, 64, 64, 150, 2)):
        m, t, ids = mesh_case(cfg, planned=True, sizes=sizes)
        with pytest.raises(bs.BSError):
            bs.bs_apply_diag(t, x, d, dev(np.zeros(cfg.NG)))
    m, t, ids = mesh_case(cfg, planned=False)
    with pytest.raises(bs.BSError):
        bs.bs_apply_diag(t, x, d, dev(np.zeros(cfg.NG)))


def test_injected_faults_are_reported(monkeypatch):
    """BS_FAULT=launch: calls report BS_ECUDA and launch nothing; a mesh built
    under BS_FAULT=badtable has out-of-range entries, which the one-pass
    kernels skip and report.  The context keeps working afterwards."""
    x, y = dev(np.arange(8.0)), dev(np.zeros(8))
    monkeypatch.setenv("BS_FAULT", "launch")
    with pytest.raises(bs.BSError) as e:
        bs.bs_copy(x, y)
    assert e.value.status == bs.BS_ECUDA
    assert bs.default_context().device_status() == bs.BS_OK
    assert np.all(host(y) == 0.0)
    cfg = gen.WORKLOADS["tiny"]
    monkeypatch.setenv("BS_FAULT", "badtable")
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    monkeypatch.delenv("BS_FAULT")
    assert m.validate() == bs.BS_EBOUNDS
    t = m.to_device(0, planned=False)
    qLd = dev(np.zeros(cfg.NL))
    bs.bs_scatter(t, dev(gen.uniform_pm1(1, 1, cfg.NG)), qLd)
    assert bs.default_context().device_status() == bs.BS_EBOUNDS
    bs.bs_gather(t, qLd, dev(np.zeros(cfg.NG)))
    assert bs.default_context().device_status() == bs.BS_EBOUNDS
    bs.bs_copy(x, y)
    assert np.array_equal(host(y), np.arange(8.0))


def test_small_planned_meshes_may_take_the_one_pass_kernels(monkeypatch):
    """With the library default, a plan on an L2-sized mesh runs the one-pass
    kernels; the results are the same bits either way."""
    monkeypatch.setenv("BS_TUNE_ONEPASS", "1")
    ctx = bs.Context(0)
    for cfg in (gen.WORKLOADS["tiny"], gen.WORKLOADS["mid"]):
        m, t, ids = mesh_case(cfg, planned=True)
        qG = gen.uniform_pm1(cfg.seed, gen.TAG_U, cfg.NG)
        qL = gen.uniform_pm1(cfg.seed, gen.TAG_P, cfg.NL)
        qLd, qGd = dev(np.zeros(cfg.NL)), dev(np.zeros(cfg.NG))
        bs.bs_scatter(t, dev(qG), qLd, ctx=ctx)
        assert bits_equal(host(qLd), oracle.scatter(ids, qG))
        bs.bs_gather(t, dev(qL), qGd, ctx=ctx)
        assert bits_equal(host(qGd), oracle.gather(ids, qL, cfg.NG))
        assert ctx.device_status() == bs.BS_OK
