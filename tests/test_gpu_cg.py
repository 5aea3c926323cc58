"""GPU parity of the device-side CG solve (bs_cg_solve) and of the AXPY
with a device-side beta (bs_axpy_dev), through the C ABI, against the
oracle's textbook CG (oracle.cg_solve).

Tolerance.  Every vector operation of an iteration is bit-exact given its
scalars (scatter/gather, the fused diagonal operator, BS5's x and r,
AXPY); the scalars rr_k = r.r and pAp_k = p.Ap are reductions.  Here every
one is a sum of non-negative terms (the operator is diagonal and positive),
for which the device reductions are within 3.2e-14 relative of the exact
sum by construction: squares in float-float with <= 2^-45 relative error
each, binary64 fma accumulation of at most a few hundred positive terms
per thread, then a tree of partials.  CG amplifies its scalars' rounding:
on the N = 5 test mesh the oracle's own x after 12 iterations moves by
2e-8 relative when its Dot2 sums are swapped for plain sequential ones.
So the bound is measured, not guessed: the oracle's iteration is re-run
with every alpha_k and beta_k scaled by 1 +- 1e-13 (two sign patterns),
and the device's x, r and scalar histories must lie within twice the
largest excursion of those runs (plus 1e-13 relative) -- tight in the
first iterations, wider as CG's sensitivity grows.  Further, the device's
recursive residual must equal b - A x of its own x to 1e-11 |b|, and its
last rr must equal r.r of its own r to 1e-12.

That holds while the Krylov space is not exhausted.  The operator is
diagonal with few distinct values (4 for the identity, 10 for the N = 3
mass, 20 for N = 5, 35 for the N = 7 mid mesh), and CG ends in that many
steps in exact arithmetic; at that step finite-precision CG's residual is
what its loss of orthogonality left (~1e-6 |r_0| for the oracle itself),
which depends on the order of every rounding.  Parity cases therefore stop
at least two steps before that count, and runs past it are checked against
the exact solution b / diag(A) instead.
"""

import math

import numpy as np
import pytest

import bsinputs as gen
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from conftest import build_lib  # noqa: E402

build_lib()
import order_fem_cg_gb300 as bs  # noqa: E402

DEV = torch.device("cuda", 0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(DEV)


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def mesh(cfg):
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    ep, npm = gen.mesh_perms(cfg)
    ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm)
    assert np.array_equal(m.tables()["scatterIds"], ids)
    return m.to_device(0, planned=True), ids


def _apply(ids, dL, v):
    if dL is None:
        return oracle.gather(ids, oracle.scatter(ids, v), v.size)
    return oracle.apply_diag(ids, dL, v)


def envelope(ids, dL, b, x0, iters, ref, eta=1e-13):
    """Largest excursion of the oracle's iteration when each alpha_k and
    beta_k is scaled by 1 + eta s_k (s_k = +1, then (-1)^k): x, r, rr, pAp."""
    ex = er = 0.0
    err = np.zeros(iters + 1)
    epap = np.zeros(iters)
    for sign in (lambda k: 1.0, lambda k: (-1.0) ** k):
        x = np.array(x0, dtype=np.float64)
        r = oracle.axpy(-1.0, _apply(ids, dL, x), 1.0, b)
        p = oracle.copy(r)
        rr = [oracle.norm(r)]
        pap = []
        for k in range(iters):
            Ap = _apply(ids, dL, p)
            pap.append(oracle.dot(p, Ap))
            x, r, rrn = oracle.cg_update(rr[k] / pap[k] * (1 + eta * sign(k)), p, Ap, x, r)
            rr.append(rrn)
            p = oracle.axpy(1.0, r, rrn / rr[k] * (1 - eta * sign(k)), p)
        ex = max(ex, np.max(np.abs(x - ref["x"])))
        er = max(er, np.max(np.abs(r - ref["r"])))
        err = np.maximum(err, np.abs(np.array(rr) - ref["rr"]))
        epap = np.maximum(epap, np.abs(np.array(pap) - np.array(ref["pAp"]))) if iters else epap
    return ex, er, err, epap


def run(cfg, ids, t, dL, iters, x0, fused=False):
    NG = cfg.NG
    b = gen.uniform_pm1(cfg.seed, gen.TAG_R, NG)
    xd, bd = dev(x0), dev(b)
    rd, pd, Apd = (torch.empty(NG, dtype=torch.float64, device=DEV) for _ in range(3))
    dLd = dev(dL) if dL is not None else None
    if fused:
        pL = torch.empty(cfg.NL, dtype=torch.float64, device=DEV)
        scal = bs.bs_cg_solve_fused(t, dLd, bd, xd, rd, pd, Apd, pL, iters)
    else:
        scal = bs.bs_cg_solve(t, dLd, bd, xd, rd, pd, Apd, iters)
    ref = oracle.cg_solve(ids, dL, b, x0, iters)
    ex, er, err, epap = envelope(ids, dL, b, x0, iters, ref)
    s = host(scal)
    rr_ref, pap_ref = np.array(ref["rr"]), np.array(ref["pAp"])
    assert np.all(np.abs(s[:iters + 1] - rr_ref) <= 2 * err + 1e-13 * rr_ref)
    assert np.all(np.abs(s[iters + 1:] - pap_ref) <= 2 * epap + 1e-13 * np.abs(pap_ref))
    x, r = host(xd), host(rd)
    bmax = np.max(np.abs(b))
    assert np.max(np.abs(x - ref["x"])) <= 2 * ex + 1e-13 * np.max(np.abs(ref["x"]))
    assert np.max(np.abs(r - ref["r"])) <= 2 * er + 1e-13 * bmax
    # the device's recursive residual is the true residual of its own x
    diag = oracle.gather(ids, dL if dL is not None else np.ones(cfg.NL), NG)
    assert np.max(np.abs(r - (b - diag * x))) <= 1e-11 * bmax
    rr_own = math.fsum((r * r).tolist())
    assert abs(s[iters] - rr_own) <= 1e-12 * rr_own
    assert bs.default_context().device_status() == bs.BS_OK
    return s


E3N5 = gen.MeshConfig("e3n5", 3, 5, 77, gen.SHUFFLE_ELEMS | gen.PERMUTE_GLOBAL)
CASES = [                      # iters <= distinct diagonal values - 2
    (gen.WORKLOADS["tiny"], "mass", 8, False),
    (gen.WORKLOADS["tiny"], "identity", 2, False),
    (gen.WORKLOADS["tiny"], "mass", 0, False),
    (gen.WORKLOADS["tiny"], "mass", 5, True),
    (E3N5, "mass", 12, False),
    (gen.WORKLOADS["mid"], "mass", 12, False),
    (gen.WORKLOADS["mid"], "identity", 2, True),
]


@pytest.mark.parametrize("cfg,op,iters,nonzero_x0", CASES,
                         ids=lambda v: getattr(v, "name", str(v)))
def test_cg_solve_matches_oracle(cfg, op, iters, nonzero_x0):
    t, ids = mesh(cfg)
    dL = gen.mass_diagonal(cfg.E, cfg.N) if op == "mass" else None
    x0 = gen.uniform_pm1(cfg.seed, gen.TAG_X, cfg.NG) if nonzero_x0 else np.zeros(cfg.NG)
    run(cfg, ids, t, dL, iters, x0)


@pytest.mark.parametrize("cfg,op,iters,nonzero_x0", CASES,
                         ids=lambda v: getattr(v, "name", str(v)))
def test_cg_solve_fused_matches_oracle(cfg, op, iters, nonzero_x0):
    """The one-kernel solve (grid barriers) against the same oracle and bounds."""
    t, ids = mesh(cfg)
    dL = gen.mass_diagonal(cfg.E, cfg.N) if op == "mass" else None
    x0 = gen.uniform_pm1(cfg.seed, gen.TAG_X, cfg.NG) if nonzero_x0 else np.zeros(cfg.NG)
    run(cfg, ids, t, dL, iters, x0, fused=True)


@pytest.mark.parametrize("cfg,op,distinct", [(gen.WORKLOADS["tiny"], "identity", 4),
                                             (gen.WORKLOADS["tiny"], "mass", 10)],
                         ids=lambda v: getattr(v, "name", str(v)))
def test_cg_solve_reaches_the_exact_solution(cfg, op, distinct):
    """Past the distinct-eigenvalue count the device iterate is b / diag(A)
    (Z^T diag(d) Z is diagonal: entry g sums d over g's local copies)."""
    t, ids = mesh(cfg)
    NG = cfg.NG
    dL = gen.mass_diagonal(cfg.E, cfg.N) if op == "mass" else np.ones(cfg.NL)
    diag = oracle.gather(ids, dL, NG)
    assert np.unique(np.round(diag / diag.max(), 12)).size == distinct
    b = gen.uniform_pm1(cfg.seed, gen.TAG_R, NG)
    xd = torch.zeros(NG, dtype=torch.float64, device=DEV)
    rd, pd, Apd = (torch.empty(NG, dtype=torch.float64, device=DEV) for _ in range(3))
    xs = b / diag
    for fused in (False, True):
        xd.zero_()
        dLd = dev(dL) if op == "mass" else None
        if fused:
            pL = torch.empty(cfg.NL, dtype=torch.float64, device=DEV)
            scal = host(bs.bs_cg_solve_fused(t, dLd, dev(b), xd, rd, pd, Apd, pL, distinct + 2))
        else:
            scal = host(bs.bs_cg_solve(t, dLd, dev(b), xd, rd, pd, Apd, distinct + 2))
        assert np.max(np.abs(host(xd) - xs)) <= 1e-7 * np.max(np.abs(xs)), fused
        assert scal[distinct + 2] < 1e-8 * scal[0], fused
        assert bs.default_context().device_status() == bs.BS_OK


def test_cg_solve_graph_replay_is_bitwise_eager():
    """The whole solve never synchronises: it captures into one CUDA graph,
    whose replay gives the eager result bit for bit."""
    cfg = gen.WORKLOADS["tiny"]
    t, ids = mesh(cfg)
    NG, iters = cfg.NG, 8
    dL = dev(gen.mass_diagonal(cfg.E, cfg.N))
    b = dev(gen.uniform_pm1(cfg.seed, gen.TAG_R, NG))
    x, r, p, Ap = (torch.zeros(NG, dtype=torch.float64, device=DEV) for _ in range(4))
    scal = torch.zeros(2 * iters + 1, dtype=torch.float64, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):      # warm-up outside capture (kernel attributes, context)
        bs.bs_cg_solve(t, dL, b, x, r, p, Ap, iters, scal, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    eager_x, eager_s = host(x).copy(), host(scal).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        x.zero_()
        bs.bs_cg_solve(t, dL, b, x, r, p, Ap, iters, scal,
                       stream=torch.cuda.current_stream())
    x.fill_(7.0)
    scal.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host(x).view(np.uint64), eager_x.view(np.uint64))
    assert np.array_equal(host(scal).view(np.uint64), eager_s.view(np.uint64))
    g.replay()
    assert np.array_equal(host(x).view(np.uint64), eager_x.view(np.uint64))


@pytest.mark.parametrize("n", [0, 1, 5, 1000, 65536 + 3])
def test_axpy_dev_matches_oracle(n):
    x = gen.uniform_pm1(3, 1, n)
    y = gen.uniform_pm1(3, 2, n)
    num, den = 0.7312, -1.9187
    sc = dev(np.array([num, den, 0.0]))
    yd = dev(y)
    bs.bs_axpy_dev(0.37, dev(x), sc[0:1], sc[1:2], yd)
    assert np.array_equal(host(yd).view(np.uint64),
                          oracle.axpy(0.37, x, num / den, y).view(np.uint64))
    yd = dev(y)                                  # zero denominator: beta = 0
    bs.bs_axpy_dev(1.0, dev(x), sc[0:1], sc[2:3], yd)
    assert np.array_equal(host(yd).view(np.uint64), oracle.axpy(1.0, x, 0.0, y).view(np.uint64))


def test_cg_solve_rejects_bad_arguments():
    cfg = gen.WORKLOADS["tiny"]
    t, ids = mesh(cfg)
    NG = cfg.NG
    v = [torch.zeros(NG, dtype=torch.float64, device=DEV) for _ in range(5)]
    with pytest.raises(bs.BSError):
        bs.bs_cg_solve(t, None, v[0], v[1], v[1], v[2], v[3], 2)      # r overlaps x
    with pytest.raises(bs.BSError):
        bs.bs_cg_solve(t, None, v[0], v[1], v[2], v[2], v[3], 2)      # r and p overlap
    big = torch.zeros(NG + 5, dtype=torch.float64, device=DEV)
    with pytest.raises(bs.BSError):
        bs.bs_cg_solve(t, None, v[0], v[1], v[2], v[3], big[:NG], 2, scal=big[NG - 1:NG + 4])
    with pytest.raises(ValueError):
        bs.bs_cg_solve(t, None, v[0], v[1], v[2], v[3], v[4], 2, scal=v[4][:3])


def test_grid_barrier_wait_is_bounded():
    """The fused solve's grid barrier: with every block present it passes;
    with one block absent the others' bounded waits run out, the kernel
    ends, the status says so, and the context keeps working."""
    assert bs.bs_probe_grid_barrier(-1) == bs.BS_OK
    assert bs.bs_probe_grid_barrier(3) == bs.BS_ETIMEOUT
    assert bs.default_context().device_status() == bs.BS_OK     # read and cleared
    assert bs.bs_probe_grid_barrier(-1) == bs.BS_OK
    x = dev(np.arange(5.0))
    assert host(bs.bs_dot(x, x))[0] == 30.0
