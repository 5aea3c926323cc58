"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each check below ties an oracle function to something the pages or the
mathematics fix independently of the oracle's code:

  * the published SplitMix64 test vector (input generator);
  * the node counts N_L = K(p+1)^3, N_G = (EN+1)^3 of the workload meshes;
  * geometric brute force: physical GLL node coordinates, deduplicated, give
    the global nodes (two locals share a global id iff they share a point);
  * the closed-form multiplicity histogram C(3,k) a^k b^(3-k);
  * gather(scatter(u)) = m * u, sum(q_G) = sum(q_L), dense Z / Z^T products;
  * closed-form norms and dots, exact rational arithmetic (Fraction) for the
    fused multiply-adds, and the Ogita-Rump-Oishi error bound for Dot2.

The last group plants mistakes in copies of oracle steps and checks that the
pins catch them.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

import bsinputs as gen
import oracle

U = 2.0 ** -53  # unit roundoff of binary64


# ----------------------------------------------------------------------------
# Independent geometry: physical coordinates of every local node.
# ----------------------------------------------------------------------------

def gll_nodes(N):
    """Gauss-Lobatto-Legendre nodes on [-1, 1]: the end points and the roots of P_N'."""
    if N == 1:
        return np.array([-1.0, 1.0])
    inner = np.sort(np.polynomial.legendre.Legendre.basis(N).deriv().roots().real)
    return np.concatenate([[-1.0], inner, [1.0]])


def cube_rotations():
    """The 24 proper rotations of the cube in the numbering's order, as
    (perm, flip): axis permutations in lexicographic order, flip masks
    0..7 (bit a: output axis a reversed), determinant +1 kept."""
    import itertools
    out = []
    for perm in itertools.permutations(range(3)):
        inv = sum(perm[a] > perm[b] for a in range(3) for b in range(a + 1, 3))
        for f in range(8):
            flip = tuple((f >> a) & 1 for a in range(3))
            if (inv + sum(flip)) % 2 == 0:
                out.append((perm, flip))
    return out


def rotation_matrix(perm, flip):
    """Linear part of the map v -> w, w_a = +-v[perm[a]]."""
    R = np.zeros((3, 3), dtype=int)
    for a in range(3):
        R[a, perm[a]] = -1 if flip[a] else 1
    return R


def local_coords(E, N, elem_perm, orient=None):
    """(x, y, z) of each local node: element lattice cell mapped to [0,1]^3,
    reference GLL node of index w = rotation(i, j, k) mapped affinely into
    it (orient[e] selects the rotation of lattice element e)."""
    r = gll_nodes(N)
    q = N + 1
    K = E ** 3
    e = np.asarray(elem_perm, dtype=np.int64)
    ex, ey, ez = e % E, (e // E) % E, e // (E * E)
    # local node n = i + q (j + q k) inside a slot, i fastest
    n = np.arange(q ** 3)
    v = np.stack([n % q, (n // q) % q, n // (q * q)])          # 3 x q^3
    rots = cube_rotations()
    o = np.zeros(K, dtype=np.int64) if orient is None else np.asarray(orient)[e].astype(np.int64)
    w = np.empty((K, 3, q ** 3), dtype=np.int64)
    for idx, (perm, flip) in enumerate(rots):
        sel = o == idx
        if sel.any():
            wa = np.stack([N - v[perm[a]] if flip[a] else v[perm[a]] for a in range(3)])
            w[sel] = wa[None]
    x = (ex[:, None] + (1.0 + r[w[:, 0]]) / 2.0) / E
    y = (ey[:, None] + (1.0 + r[w[:, 1]]) / 2.0) / E
    z = (ez[:, None] + (1.0 + r[w[:, 2]]) / 2.0) / E
    return np.stack([x.reshape(-1), y.reshape(-1), z.reshape(-1)], axis=1).reshape(K * q ** 3, 3)


def geometric_ids(E, N, elem_perm, node_perm, mask=False, orient=None):
    """Expected local-to-global table from geometry alone: the lattice number
    of a node is its rank along each axis among the distinct coordinates."""
    c = local_coords(E, N, elem_perm, orient)
    M = E * N + 1
    g = []
    for a in range(3):
        ua = np.unique(c[:, a])
        assert ua.size == M
        g.append(np.searchsorted(ua, c[:, a]))
    L = g[0] + M * (g[1] + M * g[2])
    ids = np.asarray(node_perm)[L].astype(np.int32)
    if mask:
        on_b = np.any((c == 0.0) | (c == 1.0), axis=1)
        ids[on_b] = -1
    return ids


def ids_match_geometry(E, N, elem_perm, node_perm, ids, mask=False, orient=None):
    c = local_coords(E, N, elem_perm, orient)
    _, inv = np.unique(c, axis=0, return_inverse=True)
    inv = inv.reshape(-1)
    # two local nodes share a global id iff they share a point
    pairs = set(zip(inv.tolist(), np.asarray(ids).tolist()))
    if not mask:
        if len(pairs) != (E * N + 1) ** 3 or len(set(i for i, _ in pairs)) != len(pairs):
            return False
        if len(set(g for _, g in pairs)) != len(pairs):
            return False
    return np.array_equal(np.asarray(ids), geometric_ids(E, N, elem_perm, node_perm, mask, orient))


def multiplicity_closed_form(E, N):
    a, b = E - 1, E * (N - 1) + 2
    return {2 ** k: math.comb(3, k) * a ** k * b ** (3 - k) for k in range(4)}


def mesh(cfg_or_EN, seed=12345, flags=gen.SHUFFLE_ELEMS | gen.PERMUTE_GLOBAL):
    if isinstance(cfg_or_EN, gen.MeshConfig):
        cfg = cfg_or_EN
    else:
        E, N = cfg_or_EN
        cfg = gen.MeshConfig("t", E, N, seed, flags)
    ep, npm = gen.mesh_perms(cfg)
    orient = gen.element_orientations(cfg) if cfg.flags & gen.ROTATE_ELEMS else None
    ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm, bool(cfg.flags & gen.MASK_BOUNDARY),
                                 orient)
    return cfg, ep, npm, ids


# ----------------------------------------------------------------------------
# Input generator pins
# ----------------------------------------------------------------------------

def test_splitmix64_published_vector(golden):
    expect = [int(r[0]) for r in golden("splitmix64_seed1234567.txt")]
    # tag 0 makes the stream key equal to the seed
    assert [int(v) for v in gen.draws(1234567, 0, 5)] == expect
    assert [gen.mix64_int(1234567 + (i + 1) * gen.GAMMA) for i in range(5)] == expect
    # counter-based: a window equals the corresponding slice
    assert np.array_equal(gen.draws(1234567, 0, 3, start=2), gen.draws(1234567, 0, 5)[2:])


def test_uniform_values_exact_form():
    z = gen.draws(7, 3, 2000) >> np.uint64(11)
    u = gen.uniform_pm1(7, 3, 2000)
    for k, v in zip(z.tolist(), u.tolist()):
        assert Fraction(v) == Fraction(2 * k + 1, 2 ** 53) - 1
    assert np.all(np.abs(u) < 1.0) and np.all(u != 0.0)
    assert abs(u.mean()) < 0.05


def test_permutation_definition():
    n = 3000
    keys = gen.draws(99, 1, n).tolist()
    expect = sorted(range(n), key=lambda i: (keys[i], i))
    p = gen.permutation(99, 1, n)
    assert p.tolist() == expect
    assert np.array_equal(np.sort(p), np.arange(n))


def test_normal_moments():
    v = gen.normal(5, 3, 200000)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


# ----------------------------------------------------------------------------
# Mesh numbering pins
# ----------------------------------------------------------------------------

def test_mesh_sizes(golden):
    for name, E, N, NL, NG in golden("mesh_sizes.txt"):
        cfg = gen.WORKLOADS[name]
        assert (cfg.E, cfg.N) == (int(E), int(N))
        assert cfg.NL == int(NL) and cfg.NG == int(NG)
        assert cfg.NL == cfg.K * (cfg.N + 1) ** 3


@pytest.mark.parametrize("E,N,flags", [
    (2, 2, 0), (2, 2, 3), (3, 3, 3), (2, 5, 3), (1, 1, 0), (1, 4, 3), (4, 2, 1), (3, 1, 2)])
def test_numbering_matches_geometry(E, N, flags):
    cfg, ep, npm, ids = mesh((E, N), seed=1000 + E * 10 + N, flags=flags)
    assert ids.size == cfg.NL
    assert ids.min() >= 0 and ids.max() < cfg.NG
    assert ids_match_geometry(E, N, ep, npm, ids)


@pytest.mark.parametrize("E,N", [(2, 2), (3, 3), (1, 2)])
def test_masked_numbering_matches_geometry(E, N):
    flags = gen.SHUFFLE_ELEMS | gen.PERMUTE_GLOBAL | gen.MASK_BOUNDARY
    cfg, ep, npm, ids = mesh((E, N), seed=77, flags=flags)
    assert ids_match_geometry(E, N, ep, npm, ids, mask=True)
    M = E * N + 1
    # masked globals = the box-boundary lattice nodes
    unmasked_globals = np.unique(ids[ids >= 0])
    assert unmasked_globals.size == max(M - 2, 0) ** 3


def test_rotations_form_the_cube_rotation_group():
    """The numbering's 24 orientations are exactly the rotation group of the
    cube: orthogonal, determinant +1, distinct, closed under composition,
    the identity first."""
    mats = [rotation_matrix(p, f) for p, f in cube_rotations()]
    assert len(mats) == 24 and np.array_equal(mats[0], np.eye(3, dtype=int))
    keys = {m.tobytes() for m in mats}
    assert len(keys) == 24
    for m in mats:
        assert np.array_equal(m @ m.T, np.eye(3, dtype=int)) and round(np.linalg.det(m)) == 1
    for a in mats:
        for b in mats:
            assert (a @ b).tobytes() in keys


def test_orientation_draws_definition():
    cfg = gen.MeshConfig("t", 5, 2, 99, gen.ROTATE_ELEMS)
    o = gen.element_orientations(cfg)
    z = [int(v) for v in gen.draws(99, gen.TAG_ORIENT, cfg.K)]
    assert o.tolist() == [((v >> 11) * 24) >> 53 for v in z]
    assert set(o.tolist()) <= set(range(24)) and len(set(o.tolist())) > 16
    assert not gen.element_orientations(gen.MeshConfig("t", 5, 2, 99, 3)).any()


@pytest.mark.parametrize("E,N,flags", [(2, 2, 8), (3, 3, 11), (2, 5, 15), (1, 4, 8), (3, 2, 12)])
def test_rotated_numbering_matches_geometry(E, N, flags):
    """Rotated elements still tile the box: two locals share a global id iff
    they share a point, and masked ids are exactly the boundary points."""
    cfg, ep, npm, ids = mesh((E, N), seed=300 + E * 10 + N, flags=flags)
    orient = gen.element_orientations(cfg)
    assert ids_match_geometry(E, N, ep, npm, ids, mask=bool(flags & gen.MASK_BOUNDARY),
                              orient=orient)
    if E > 1 and N > 1:
        # the rotations matter: the table differs from the unrotated one
        plain = oracle.box_scatter_ids(E, N, ep, npm, bool(flags & gen.MASK_BOUNDARY))
        assert not np.array_equal(ids, plain)
    m = oracle.gather(ids, (ids >= 0).astype(np.float64), cfg.NG)
    if not flags & gen.MASK_BOUNDARY:
        hist = dict(zip(*np.unique(m, return_counts=True)))
        assert {int(k): int(v) for k, v in hist.items()} == \
            {k: v for k, v in multiplicity_closed_form(E, N).items() if v}


def test_multiplicity_closed_form_golden(golden):
    for E, N, c1, c2, c4, c8 in golden("multiplicity.txt"):
        E, N = int(E), int(N)
        assert multiplicity_closed_form(E, N) == {1: int(c1), 2: int(c2), 4: int(c4), 8: int(c8)}


@pytest.mark.parametrize("which", ["tiny", "mid", (2, 2), (5, 4), (1, 3)])
def test_gather_of_ones_is_multiplicity(which):
    cfg, ep, npm, ids = mesh(gen.WORKLOADS[which] if isinstance(which, str) else which)
    m = oracle.gather(ids, np.ones(cfg.NL), cfg.NG)
    vals, counts = np.unique(m, return_counts=True)
    hist = dict(zip(vals.astype(int).tolist(), counts.tolist()))
    expect = {k: v for k, v in multiplicity_closed_form(cfg.E, cfg.N).items() if v}
    assert hist == expect
    assert int(m.sum()) == cfg.NL


def test_dense_Z_brute_force_2x2x2():
    """Dense 216 x 125 Boolean Z from coordinates; oracle scatter = Z q_G and
    gather = Z^T q_L, on integer data where every order is exact."""
    E, N = 2, 2
    cfg, ep, npm, ids = mesh((E, N), seed=4242)
    gids = geometric_ids(E, N, ep, npm)
    Z = np.zeros((cfg.NL, cfg.NG))
    Z[np.arange(cfg.NL), gids] = 1.0
    assert np.all(Z.sum(axis=1) == 1.0)                 # one nonzero per row of Z
    qG = gen.integers_dyadic(1, 3, cfg.NG)
    qL = gen.integers_dyadic(1, 4, cfg.NL)
    assert np.array_equal(oracle.scatter(ids, qG), Z @ qG)
    assert np.array_equal(oracle.gather(ids, qL, cfg.NG), Z.T @ qL)


@pytest.mark.parametrize("which", ["tiny", (3, 3)])
def test_gather_scatter_identities(which):
    cfg, ep, npm, ids = mesh(gen.WORKLOADS[which] if isinstance(which, str) else which)
    m = oracle.gather(ids, np.ones(cfg.NL), cfg.NG)
    u = gen.integers_dyadic(cfg.seed, gen.TAG_U, cfg.NG)
    assert np.array_equal(oracle.gather(ids, oracle.scatter(ids, u), cfg.NG), m * u)
    qL = gen.uniform_pm1(cfg.seed, gen.TAG_P, cfg.NL)
    qG = oracle.gather(ids, qL, cfg.NG)
    assert abs(math.fsum(qG) - math.fsum(qL)) <= 1e-12 * math.fsum(np.abs(qL))


def test_masked_scatter_and_gather():
    flags = gen.SHUFFLE_ELEMS | gen.PERMUTE_GLOBAL | gen.MASK_BOUNDARY
    cfg, ep, npm, ids = mesh((3, 2), seed=5, flags=flags)
    qG = gen.uniform_pm1(1, 2, cfg.NG)
    qL = oracle.scatter(ids, qG)
    assert np.all(qL[ids < 0] == 0.0) and np.all(np.signbit(qL[ids < 0]) == False)
    assert np.array_equal(qL[ids >= 0], qG[ids[ids >= 0]])
    m = oracle.gather(ids, np.ones(cfg.NL), cfg.NG)
    c = local_coords(3, 2, ep)
    interior = ~np.any((c == 0.0) | (c == 1.0), axis=1)
    g_int = np.unique(ids[interior])
    assert np.all(m[g_int] >= 1)
    rest = np.setdiff1d(np.arange(cfg.NG), g_int)
    assert np.all(m[rest] == 0.0)


def _gather_by_rows(ids, qL, NG):
    """Brute force: for each global node, its local copies sorted ascending, summed from +0.0."""
    out = []
    for g in range(NG):
        ls = np.sort(np.nonzero(ids == g)[0])
        s = 0.0
        for l in ls:
            s = s + float(qL[l])
        out.append(s)
    return np.array(out)


def order_probe(ids, NG, first_big):
    """Values whose row sum depends on order: per row, one 1.0 and 2^-53 elsewhere."""
    qL = np.full(ids.size, 2.0 ** -53)
    for g in range(NG):
        ls = np.sort(np.nonzero(ids == g)[0])
        qL[ls[0] if first_big else ls[-1]] = 1.0
    return qL


def test_gather_sum_order_is_ascending_local_index():
    cfg, ep, npm, ids = mesh((2, 2), seed=31)
    for first_big in (True, False):
        qL = order_probe(ids, cfg.NG, first_big)
        got = oracle.gather(ids, qL, cfg.NG)
        assert np.array_equal(got, _gather_by_rows(ids, qL, cfg.NG))
    qL = gen.uniform_pm1(3, 3, cfg.NL)
    assert np.array_equal(oracle.gather(ids, qL, cfg.NG), _gather_by_rows(ids, qL, cfg.NG))
    # +0.0 start: a single -0.0 contribution gives +0.0
    qL = np.full(cfg.NL, -0.0)
    assert not np.any(np.signbit(oracle.gather(ids, qL, cfg.NG)))


# ----------------------------------------------------------------------------
# Vector operation pins
# ----------------------------------------------------------------------------

def test_copy_is_bitwise_identity():
    x = np.array([0.0, -0.0, 1.5, np.inf, -np.inf, 5e-324, -2.2250738585072014e-308, 1e308])
    bits = np.concatenate([x.view(np.uint64), np.array([0x7FF8000000000123, 0xFFF0000000000001],
                                                        dtype=np.uint64)])
    x = bits.view(np.float64)
    assert np.array_equal(oracle.copy(x).view(np.uint64), bits)
    assert oracle.copy(np.zeros(0)).size == 0


def _round(fr):
    return float(fr)   # CPython int/int true division rounds correctly (ties to even)


@pytest.mark.parametrize("beta", [1.0, -0.5, 0.3])
def test_axpy_matches_exact_rational(beta):
    n = 3000
    x = gen.uniform_pm1(11, 1, n) * 1e3
    y = gen.uniform_pm1(11, 2, n)
    alpha = 0.37
    got = oracle.axpy(alpha, x, beta, y)
    for i in range(n):
        by = _round(Fraction(beta) * Fraction(y[i]))    # beta * y_i rounded first
        assert got[i] == _round(Fraction(alpha) * Fraction(x[i]) + Fraction(by))


def test_cg_update_matches_exact_rational():
    n = 2000
    p, Ap, x, r = (gen.uniform_pm1(21, t, n) for t in (4, 5, 7, 6))
    alpha = 0.6180339887
    x1, r1, rr = oracle.cg_update(alpha, p, Ap, x, r)
    for i in range(n):
        assert x1[i] == _round(Fraction(alpha) * Fraction(p[i]) + Fraction(x[i]))
        assert r1[i] == _round(-Fraction(alpha) * Fraction(Ap[i]) + Fraction(r[i]))
    exact = sum(Fraction(v) * Fraction(v) for v in r1.tolist())
    assert abs(Fraction(rr) - exact) <= 2 * U * exact


def test_norm_closed_forms():
    n = 1000003
    assert oracle.norm(np.full(n, 0.5)) == n / 4
    n = 100003
    i = np.arange(n, dtype=np.float64)
    exact = (n - 1) * n * (2 * n - 1) // 6
    assert abs(Fraction(oracle.norm(i)) - exact) <= U * exact
    assert oracle.dot(i, np.ones(n)) == n * (n - 1) // 2
    assert oracle.norm(np.zeros(0)) == 0.0 and not math.copysign(1.0, oracle.norm(np.zeros(0))) < 0


def ill_conditioned_pair(n, seed):
    """x, y whose exact dot is tiny next to sum |x_i y_i|: the last term cancels the rest."""
    x = gen.uniform_pm1(seed, 1, n)
    y = gen.uniform_pm1(seed, 2, n)
    s = math.fsum(x[:-1] * y[:-1])
    x[-1] = 1.0
    y[-1] = -s
    return x, y


def _exact_dot(x, y):
    return sum(Fraction(a) * Fraction(b) for a, b in zip(x.tolist(), y.tolist()))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_dot2_error_bound(seed):
    """Ogita-Rump-Oishi: |Dot2 - s| <= u|s| + gamma_n^2 sum|x_i y_i|; the plain
    sum only meets gamma_n sum|x_i y_i|."""
    n = 4000
    x, y = ill_conditioned_pair(n, seed)
    s = _exact_dot(x, y)
    absum = sum(abs(Fraction(a) * Fraction(b)) for a, b in zip(x.tolist(), y.tolist()))
    g = n * U / (1 - n * U)
    d2 = Fraction(oracle.dot(x, y))
    assert abs(d2 - s) <= U * abs(s) + Fraction(g * g) * absum
    dp = Fraction(oracle.dot_plain(x, y))
    assert abs(dp - s) <= Fraction(g) * absum


# ----------------------------------------------------------------------------
# Planted mistakes: copies of oracle steps with one plausible error each must
# fail the pins above.
# ----------------------------------------------------------------------------

def _ids_ij_swapped(E, N, ep, npm):
    ids = oracle.box_scatter_ids(E, N, ep, npm)
    q = N + 1
    return ids.reshape(-1, q, q, q).transpose(0, 1, 3, 2).reshape(-1).copy()


def _ids_wrong_element_axis(E, N, ep, npm):
    # element number read as ez + E(ey + E ex)
    e = np.asarray(ep)
    ep2 = (e // (E * E)) + E * (((e // E) % E) + E * (e % E))
    return oracle.box_scatter_ids(E, N, ep2.astype(np.int32), npm)


def test_planted_numbering_mistakes_are_caught():
    E, N = 3, 2
    cfg, ep, npm, ids = mesh((E, N), seed=8)
    assert ids_match_geometry(E, N, ep, npm, ids)
    assert not ids_match_geometry(E, N, ep, npm, _ids_ij_swapped(E, N, ep, npm))
    assert not ids_match_geometry(E, N, ep, npm, _ids_wrong_element_axis(E, N, ep, npm))
    # node permutation applied in the inverse direction
    inv = np.empty_like(npm)
    inv[npm] = np.arange(npm.size, dtype=np.int32)
    bad = oracle.box_scatter_ids(E, N, ep, inv)
    assert not ids_match_geometry(E, N, ep, npm, bad)


def test_planted_gather_mistakes_are_caught():
    cfg, ep, npm, ids = mesh((2, 2), seed=31)
    qL = order_probe(ids, cfg.NG, first_big=True)
    expect = _gather_by_rows(ids, qL, cfg.NG)
    # descending local order
    desc = np.zeros(cfg.NG)
    for l in range(cfg.NL - 1, -1, -1):
        desc[ids[l]] += qL[l]
    assert not np.array_equal(desc, expect)
    # dropped last local entry, seen on generic data
    qL = gen.uniform_pm1(3, 3, cfg.NL)
    drop = oracle.gather(ids[:-1], qL[:-1], cfg.NG)
    assert not np.array_equal(drop, _gather_by_rows(ids, qL, cfg.NG))


def test_planted_reduction_mistakes_are_caught():
    n = 4000
    x, y = ill_conditioned_pair(n, 1)
    s = _exact_dot(x, y)
    absum = sum(abs(Fraction(a) * Fraction(b)) for a, b in zip(x.tolist(), y.tolist()))
    g = n * U / (1 - n * U)
    bound = U * abs(s) + Fraction(g * g) * absum
    # Dot2 without the TwoProduct error term: only the TwoSum half
    p = q = 0.0
    for a, b in zip(x.tolist(), y.tolist()):
        h = a * b
        t = p + h
        z = t - p
        q += (p - (t - z)) + (h - z)
        p = t
    assert abs(Fraction(p + q) - s) > bound
    # the plain sum
    assert abs(Fraction(oracle.dot_plain(x, y)) - s) > bound


def test_planted_axpy_mistake_is_caught():
    n = 3000
    x = gen.uniform_pm1(11, 1, n) * 1e3
    y = gen.uniform_pm1(11, 2, n)
    alpha = 0.37
    exact = [_round(Fraction(alpha) * Fraction(a) + Fraction(b)) for a, b in zip(x, y)]
    unfused = alpha * x + y          # two roundings instead of one fma
    assert not np.array_equal(unfused, np.array(exact))
    assert np.array_equal(oracle.axpy(alpha, x, 1.0, y), np.array(exact))


# ----------------------------------------------------------------------------
# Diagonal local operator (mass matrix) pins
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 3, 5, 7])
def test_gll_quadrature_exact_to_degree_2N_minus_1(N):
    """GLL quadrature integrates polynomials of degree <= 2N-1 exactly
    ("GPU accelerated spectral finite elements on all-hex meshes")."""
    x, w = gen.gll_nodes_weights(N)
    assert abs(w.sum() - 2.0) < 1e-14
    for k in range(2 * N):
        exact = 0.0 if k % 2 else 2.0 / (k + 1)
        assert abs(float(np.sum(w * x ** k)) - exact) < 1e-13
    # and not beyond (degree 2N has a quadrature error)
    assert abs(float(np.sum(w * x ** (2 * N))) - 2.0 / (2 * N + 1)) > 1e-6


def _check_mass_operator(apply, cfg, ids):
    d = gen.mass_diagonal(cfg.E, cfg.N)
    one = apply(ids, d, np.ones(cfg.NG))
    assert abs(math.fsum(one) - 1.0) < 1e-12          # total volume of [0,1]^3
    if not (cfg.flags & gen.MASK_BOUNDARY):
        assert np.all(one > 0)
    x = gen.uniform_pm1(5, 1, cfg.NG)
    y = gen.uniform_pm1(5, 2, cfg.NG)
    xy = math.fsum(x * apply(ids, d, y))
    yx = math.fsum(y * apply(ids, d, x))
    assert abs(xy - yx) <= 1e-12 * math.fsum(np.abs(x) * apply(ids, d, np.abs(y)))


@pytest.mark.parametrize("which", ["tiny", (3, 2), (2, 5)])
def test_mass_operator_volume_and_symmetry(which):
    cfg, ep, npm, ids = mesh(gen.WORKLOADS[which] if isinstance(which, str) else which)
    _check_mass_operator(oracle.apply_diag, cfg, ids)
    # with d = 1 the operator is gather(scatter(.)) = multiplicity * u
    u = gen.integers_dyadic(3, 3, cfg.NG)
    m = oracle.gather(ids, np.ones(cfg.NL), cfg.NG)
    assert np.array_equal(oracle.apply_diag(ids, np.ones(cfg.NL), u), m * u)


def test_planted_mass_operator_mistakes_are_caught():
    cfg, ep, npm, ids = mesh((3, 2))
    mutants = [
        lambda ids_, d, x: oracle.gather(ids_, oracle.scatter(ids_, x), cfg.NG),          # no d
        lambda ids_, d, x: oracle.gather(ids_, d * d * oracle.scatter(ids_, x), cfg.NG),  # d twice
        lambda ids_, d, x: oracle.gather(ids_, d * np.roll(oracle.scatter(ids_, x), 1),   # off by one
                                         cfg.NG),
    ]
    for wrong in mutants:
        with pytest.raises(AssertionError):
            _check_mass_operator(wrong, cfg, ids)


# ----------------------------------------------------------------------------
# Conjugate gradients (textbook iteration on Z^T diag(d) Z)
# ----------------------------------------------------------------------------
# Z^T diag(d) Z is diagonal (entry g: the sum of d over the local copies of
# node g), so the exact solution is b / gather(d), and CG on it terminates
# in as many steps as the diagonal has distinct values (with nonzero b
# components): facts of the method, not of the oracle's code.

def _cg_mesh(E=3, N=3, seed=12345):
    cfg = gen.MeshConfig("t", E, N, seed, gen.SHUFFLE_ELEMS | gen.PERMUTE_GLOBAL)
    ep, npm = gen.mesh_perms(cfg)
    return cfg, oracle.box_scatter_ids(E, N, ep, npm)


def test_cg_identity_operator_terminates_in_four_steps():
    """Z^T Z = diag(multiplicity), multiplicities {1, 2, 4, 8}: four steps."""
    cfg = gen.WORKLOADS["tiny"]
    ep, npm = gen.mesh_perms(cfg)
    ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm)
    m = oracle.gather(ids, np.ones(cfg.NL), cfg.NG)
    assert sorted(np.unique(m).tolist()) == [1.0, 2.0, 4.0, 8.0]
    b = gen.uniform_pm1(cfg.seed, gen.TAG_R, cfg.NG)
    res = oracle.cg_solve(ids, None, b, np.zeros(cfg.NG), 4)
    rr = np.array(res["rr"])
    assert np.all(rr[:4] > 1e-6 * rr[0]) and rr[4] < 1e-28 * rr[0]
    assert np.max(np.abs(res["x"] - b / m)) <= 1e-14 * np.max(np.abs(b))


def test_cg_mass_operator_terminates_at_distinct_eigenvalue_count():
    cfg, ids = _cg_mesh(3, 3)
    d = gen.mass_diagonal(cfg.E, cfg.N)
    diag = oracle.gather(ids, d, cfg.NG)
    nd = np.unique(np.round(diag / diag.max(), 12)).size
    assert nd == 10
    b = gen.uniform_pm1(7, 1, cfg.NG)
    res = oracle.cg_solve(ids, d, b, np.zeros(cfg.NG), nd + 1)
    rr = np.array(res["rr"])
    assert np.all(rr[:nd] > 1e-7 * rr[0]) and rr[nd] < 1e-8 * rr[0]
    xs = b / diag
    assert np.max(np.abs(res["x"] - xs)) <= 1e-9 * np.max(np.abs(xs))


def _check_cg(solve, iters=8, E=3, N=3, x0_seed=None):
    """Textbook CG properties of solve(ids, d, b, x0, k) for k = 0..iters on the
    mass operator: the recursive residual is b - A x_k, residuals are mutually
    orthogonal, directions A-conjugate (both up to the slow loss of
    orthogonality of finite-precision CG, ~1e-8 here; a wrong step breaks
    them at O(1)), the A-norm error decreases and obeys
    2 ((sqrt(kappa) - 1) / (sqrt(kappa) + 1))^k, and rr_k = r_k . r_k."""
    cfg, ids = _cg_mesh(E, N)
    d = gen.mass_diagonal(cfg.E, cfg.N)
    diag = oracle.gather(ids, d, cfg.NG)
    b = gen.uniform_pm1(7, 1, cfg.NG)
    x0 = np.zeros(cfg.NG) if x0_seed is None else gen.uniform_pm1(x0_seed, 2, cfg.NG)
    xs = b / diag
    kappa = diag.max() / diag.min()
    rho = (math.sqrt(kappa) - 1) / (math.sqrt(kappa) + 1)
    runs = [solve(ids, d, b, x0, k) for k in range(iters + 1)]
    err = [math.sqrt(math.fsum(diag * (xs - r_["x"]) ** 2)) for r_ in runs]
    bmax = np.max(np.abs(b))
    for k, r_ in enumerate(runs):
        true_r = b - diag * r_["x"]
        assert np.max(np.abs(true_r - r_["r"])) <= 1e-12 * bmax, k
        assert abs(r_["rr"][k] - math.fsum(r_["r"] ** 2)) <= 1e-13 * r_["rr"][k], k
        assert err[k] <= 2 * rho ** k * err[0] * (1 + 1e-9), k
        if k:
            assert err[k] <= err[k - 1] * (1 + 1e-12), k
    R = [r_["r"] for r_ in runs]
    P = [r_["p"] for r_ in runs]
    for i in range(iters + 1):
        for j in range(i + 1, iters + 1):
            ri, rj = math.fsum(R[i] ** 2), math.fsum(R[j] ** 2)
            assert abs(math.fsum(R[i] * R[j])) <= 1e-6 * math.sqrt(ri * rj), (i, j)
            pi, pj = math.fsum(diag * P[i] ** 2), math.fsum(diag * P[j] ** 2)
            assert abs(math.fsum(P[i] * diag * P[j])) <= 1e-6 * math.sqrt(pi * pj), (i, j)


def test_cg_textbook_properties():
    _check_cg(oracle.cg_solve)
    _check_cg(oracle.cg_solve, iters=5, x0_seed=11)


def _cg_mutant(which):
    """The textbook loop rebuilt from oracle steps with one planted mistake."""
    def solve(ids, d, b, x0, iters):
        NG = b.size
        A = lambda v: oracle.apply_diag(ids, d, v)                     # noqa: E731
        x = np.array(x0, dtype=np.float64)
        r = oracle.axpy(-1.0, A(x), 1.0, b)
        p = oracle.copy(r)
        rr = [oracle.norm(r)]
        for k in range(iters):
            Ap = A(p)
            pAp = oracle.dot(p, Ap)
            alpha = rr[k] / pAp if which != "alpha_inverted" else pAp / rr[k]
            if which == "x_along_r":
                x = oracle.axpy(alpha, r, 1.0, x)
                r = oracle.axpy(-alpha, Ap, 1.0, r)
                rrn = oracle.norm(r)
            else:
                x, r, rrn = oracle.cg_update(alpha, p, Ap, x, r)
            if which == "r_sign":
                r = oracle.axpy(2 * alpha, Ap, 1.0, r)
                rrn = oracle.norm(r)
            rr.append(rrn)
            beta = {"beta_inverted": rr[k] / rrn, "no_beta": 0.0}.get(which, rrn / rr[k])
            p = oracle.axpy(1.0, r, beta if which != "p_minus" else -beta, p)
        assert len(rr) == iters + 1 and NG == x.size
        return dict(x=x, r=r, p=p, rr=rr)
    return solve


@pytest.mark.parametrize("which", ["alpha_inverted", "x_along_r", "r_sign", "beta_inverted",
                                   "no_beta", "p_minus"])
def test_planted_cg_mistakes_are_caught(which):
    with pytest.raises(AssertionError):
        _check_cg(_cg_mutant(which), iters=6)


def test_cg_mutant_harness_without_mistake_passes():
    _check_cg(_cg_mutant("none"), iters=6)


# ----------------------------------------------------------------------------
# One CG iteration's streaming sequence (identity local operator)
# ----------------------------------------------------------------------------

def test_cg_sequence_zero_denominator_keeps_x_and_r():
    """p = 0 makes p.Ap = 0; the reading takes alpha = 0 there (a vanishing
    p.Ap occurs only at an exact solution), so x and r come back bit for bit
    and both r.r sums are the exact sum of squares (dyadic r)."""
    cfg, _, _, ids = mesh((3, 3))
    NG = cfg.NG
    pG = np.zeros(NG)
    xG = gen.uniform_pm1(61, 1, NG)
    rG = np.round(gen.uniform_pm1(61, 2, NG) * 64) / 8   # multiples of 1/8, |r| <= 8
    rG[rG == 0] = 0.125                                    # no signed zeros
    out = oracle.cg_sequence(ids, pG, xG, rG, rr=3.5)
    assert out["pAp"] == 0.0 and out["alpha"] == 0.0
    assert np.array_equal(out["x"].view(np.uint64), xG.view(np.uint64))
    assert np.array_equal(out["r"].view(np.uint64), rG.view(np.uint64))
    exact = sum(Fraction(v) ** 2 for v in rG.tolist())
    assert Fraction(out["rr_new"]) == exact and Fraction(out["rnorm"]) == exact


def test_cg_sequence_exact_on_small_integers():
    """With small-integer p, x, r every step is exact: Z^T Z p = m p with m the
    node multiplicity (counted here with bincount, not with the oracle's
    gather), p.Ap = sum m p^2; rr = 2 p.Ap gives alpha = 2 exactly, so
    x + 2p, r - 2 m p and their squares are exact integers."""
    cfg, _, _, ids = mesh((3, 3))
    NG = cfg.NG
    m = np.bincount(ids[ids >= 0], minlength=NG).astype(np.int64)
    pi = np.round(gen.uniform_pm1(62, 1, NG) * 7).astype(np.int64)
    xi = np.round(gen.uniform_pm1(62, 2, NG) * 50).astype(np.int64)
    ri = np.round(gen.uniform_pm1(62, 3, NG) * 50).astype(np.int64)
    pAp = int(np.sum(m * pi * pi))
    assert 0 < pAp < 2 ** 52
    out = oracle.cg_sequence(ids, pi.astype(float), xi.astype(float), ri.astype(float),
                             rr=float(2 * pAp))
    assert np.array_equal(out["pL"], pi[ids].astype(float))
    assert np.array_equal(out["ApG"], (m * pi).astype(float))
    assert out["pAp"] == pAp and out["alpha"] == 2.0
    assert np.array_equal(out["x"], (xi + 2 * pi).astype(float))
    r1 = ri - 2 * m * pi
    assert np.array_equal(out["r"], r1.astype(float))
    assert out["rr_new"] == int(np.sum(r1 * r1)) == out["rnorm"]
