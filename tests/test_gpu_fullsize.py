"""Parity at full size: the stress mesh (56,623,104 local / 33,076,161 global
nodes) in exactly the configuration bench.py times, every output of one step
compared with the oracle on the whole arrays (bit-exact, or 1e-12 relative
for the reductions)."""

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
import bench  # noqa: E402
import order_fem_cg_gb300 as bs  # noqa: E402


def same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint64), np.asarray(b).view(np.uint64))


def close(a, b, rtol=1e-12):
    return abs(a - b) <= rtol * abs(b)


@pytest.mark.parametrize("name,planned", [("stress", True), ("stress", False),
                                          ("stress_masked", True)])
def test_stress_step_matches_oracle(name, planned):
    """The stress mesh, and the same scale with masked boundary nodes and
    randomly oriented elements."""
    cfg = gen.WORKLOADS[name]
    torch.cuda.set_device(0)
    wl = bench.Workload(cfg, torch, bs, torch.device("cuda", 0), planned=planned)
    assert wl.planned == planned
    h, v, sc = wl.h, wl.v, wl.sc
    ids = oracle_ids(cfg)
    assert np.array_equal(wl.mesh.tables()["scatterIds"], ids)
    stream = torch.cuda.current_stream()
    for name in wl.names:
        wl.op(name, stream)
    torch.cuda.synchronize()

    def g(k):
        return v[k].cpu().numpy()

    def s(k):
        return sc[k].cpu().item()

    assert same(g("b"), h["u"])
    assert same(g("d"), oracle.axpy(cfg.alpha, h["p"], cfg.beta, h["r"]))
    assert close(s("norm"), oracle.norm(h["Ap"]))
    assert close(s("dot"), oracle.dot(h["x"], h["u"]))
    xo, ro, rro = oracle.cg_update(cfg.alpha, h["p"], h["Ap"], h["x"], h["r"])
    assert same(g("X"), xo) and same(g("R"), ro) and close(s("rdotr"), rro)
    del xo, ro
    assert same(g("qG1"), oracle.gather(ids, h["u"], cfg.NG))
    assert same(g("qL2"), oracle.scatter(ids, h["qG"]))
    ref = oracle.cg_sequence(ids, h["pG"], h["xG"], h["rG"], wl.rr_host)
    assert same(g("pL"), ref["pL"]) and same(g("ApG"), ref["ApG"])
    assert close(s("pAp"), ref["pAp"])
    da = 2e-12 * abs(ref["alpha"])
    xg, rg = g("xG"), g("rG")
    assert np.all(np.abs(xg - ref["x"]) <= da * np.abs(h["pG"]) + np.spacing(np.abs(ref["x"])))
    assert np.all(np.abs(rg - ref["r"]) <= da * np.abs(ref["ApG"]) + np.spacing(np.abs(ref["r"])))
    assert close(s("rnorm"), oracle.norm(rg))
    assert bs.default_context().device_status() == bs.BS_OK


def test_stress_mass_operator_and_cg_solve():
    """The fused global operator Z^T diag(d) Z (GLL mass) on the stress mesh,
    bit-exact against the oracle, and three CG iterations of both solves
    within the oracle's envelope under 1e-13 perturbations of its scalars
    (see test_gpu_cg.py for the bound)."""
    from test_gpu_cg import envelope

    cfg = gen.WORKLOADS["stress"]
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    m = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    t = m.to_device(0)
    ids = oracle_ids(cfg)
    NG = cfg.NG
    dL = gen.mass_diagonal(cfg.E, cfg.N)
    x = gen.uniform_pm1(cfg.seed, gen.TAG_X, NG)
    dLd = torch.from_numpy(dL).to(dev)
    y = torch.empty(NG, dtype=torch.float64, device=dev)
    bs.bs_apply_diag(t, torch.from_numpy(x).to(dev), dLd, y)
    assert same(y.cpu().numpy(), oracle.apply_diag(ids, dL, x))
    del y
    b = gen.uniform_pm1(cfg.seed, gen.TAG_R, NG)
    iters = 3
    ref = oracle.cg_solve(ids, dL, b, np.zeros(NG), iters)
    ex, er, err, epap = envelope(ids, dL, b, np.zeros(NG), iters, ref)
    for fused in (False, True):
        xd, rd, pd, Apd = (torch.zeros(NG, dtype=torch.float64, device=dev) for _ in range(4))
        bd = torch.from_numpy(b).to(dev)
        if fused:
            pL = torch.empty(cfg.NL, dtype=torch.float64, device=dev)
            s = bs.bs_cg_solve_fused(t, dLd, bd, xd, rd, pd, Apd, pL, iters).cpu().numpy()
            del pL
        else:
            s = bs.bs_cg_solve(t, dLd, bd, xd, rd, pd, Apd, iters).cpu().numpy()
        xs, rs = xd.cpu().numpy(), rd.cpu().numpy()
        assert np.all(np.abs(s[:iters + 1] - ref["rr"]) <= 2 * err + 1e-13 * np.array(ref["rr"]))
        assert np.max(np.abs(xs - ref["x"])) <= 2 * ex + 1e-13 * np.max(np.abs(ref["x"]))
        assert np.max(np.abs(rs - ref["r"])) <= 2 * er + 1e-13 * np.max(np.abs(b))
        assert bs.default_context().device_status() == bs.BS_OK
        del xd, rd, pd, Apd, bd
