"""Pins of the streaming performance model (eqs. (8)-(10)) and byte counts."""

import numpy as np
import pytest

import bsinputs as gen
from order_fem_cg_gb300 import perfmodel as pm


def test_fischer_brown_point_solves_eq9():
    """B_0.8 = 4 T0 Wmax is where W_eff reaches 0.8 Wmax (bisection on eq. (9))."""
    for T0, W in [(5e-6, 7e12), (2.5e-5, 9e11), (1e-6, 3e11)]:
        lo, hi = 1.0, 1e15
        for _ in range(200):
            mid = (lo * hi) ** 0.5
            if pm.w_eff(mid, T0, W) < 0.8 * W:
                lo = mid
            else:
                hi = mid
        assert abs(hi / pm.b_08(T0, W) - 1) < 1e-9
        assert pm.w_eff(pm.b_08(T0, W), T0, W) == pytest.approx(0.8 * W, rel=1e-12)


def test_fit_recovers_parameters():
    B = np.array([2.0 ** k for k in range(13, 31)])
    T0, W = 4.2e-6, 6.5e12
    T = pm.t_model(B, T0, W)
    t0, w = pm.fit(B, T)
    assert t0 == pytest.approx(T0, rel=1e-6) and w == pytest.approx(W, rel=1e-6)
    # the model is monotone and tends to Wmax
    assert pm.w_eff(1e15, T0, W) == pytest.approx(W, rel=1e-3)


def test_byte_counts_of_the_workload_meshes():
    st = gen.WORKLOADS["stress"]
    NL, NG = st.NL, st.NG
    assert pm.bytes_scatter(NL, NG) == 944_086_536
    assert pm.bytes_gather(NL, NG, NL, 0) - 4 - 4 == 1_076_391_180
    assert pm.bytes_copy(NL) == 16 * 56_623_104
    tiny = gen.WORKLOADS["tiny"]
    assert pm.bytes_scatter(tiny.NL, tiny.NG) == 518_216
    lg = gen.WORKLOADS["large"]
    seq = pm.bytes_cg_iteration(lg.NL, lg.NG, lg.NL, 0) - 4 - 4
    assert seq == 24 * lg.NL + 92 * lg.NG


def test_moved_bytes_of_the_two_pass_design():
    """The two-pass gather and scatter route every entry through the work
    array (8 bytes written, 8 read, a 16-bit offset each way); their ceiling
    on the stress mesh is the algorithmic / moved ratio."""
    import bsinputs as gen
    c = gen.WORKLOADS["stress"]
    NL, NG = c.NL, c.NG
    assert pm.moved_bytes("gather", NL, NG, NL) == 8 * NL + 20 * NL + 10 * NG
    assert pm.moved_bytes("scatter", NL, NG, NL) == 8 * NG + 20 * NL + 8 * NL
    for op, n in (("copy", 16), ("axpy", 24), ("norm", 8), ("dot", 16), ("cg_update", 48)):
        assert pm.moved_bytes(op, NL, NG, NL) == n * NL
    g = pm.bytes_gather(NL, NG, NL, 0) / pm.moved_bytes("gather", NL, NG, NL)
    s = pm.bytes_scatter(NL, NG) / pm.moved_bytes("scatter", NL, NG, NL)
    assert abs(g - 0.562) < 0.001 and abs(s - 0.510) < 0.001
