"""CPU oracle for the Benchmark Streaming operations -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
(``bench.py``: ``cpu_baseline`` and ``--impl reference``) may import this
package.  The library (``order_fem_cg_gb300``) never does, and the oracle
never imports the library: the two share only the seeded inputs of
``bsinputs``.

Every operation is a plain loop in ``oracle.c`` (binary64, explicit fma,
-ffp-contract=off), wrapped here with numpy for argument marshalling.  The
sources each function follows are cited in ``oracle.c``:

  * "Portable high-order finite element kernels I: Streaming Operations"
    (the BS1-BS7 definitions, eq. (3), the gather/scatter kernel text);
  * "GPU accelerated spectral finite elements on all-hex meshes"
    (local-to-global and global-to-local tables);
  * Ogita, Rump, Oishi (2005), Dot2, for the accurate reductions.

Pins (checked by ``tests/test_oracle_pins.py`` against facts fixed by the
pages and by mathematics, not against this code): every function below is
pinned; none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_dbl = ctypes.c_double

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_copy.argtypes = [_i64, _f64p, _f64p]
        lib.oracle_axpy.argtypes = [_i64, _dbl, _f64p, _dbl, _f64p]
        lib.oracle_dot_plain.argtypes = [_i64, _f64p, _f64p]
        lib.oracle_dot_plain.restype = _dbl
        lib.oracle_dot2.argtypes = [_i64, _f64p, _f64p]
        lib.oracle_dot2.restype = _dbl
        lib.oracle_cg_update.argtypes = [_i64, _dbl, _f64p, _f64p, _f64p, _f64p]
        lib.oracle_scatter.argtypes = [_i64, _i32p, _f64p, _f64p]
        lib.oracle_gather.argtypes = [_i64, _i64, _i32p, _f64p, _f64p]
        lib.oracle_box_scatter_ids.argtypes = [ctypes.c_int, ctypes.c_int, _i32p, _i32p,
                                               ctypes.c_int, ctypes.c_void_p, _i32p]
        for f in (lib.oracle_copy, lib.oracle_axpy, lib.oracle_cg_update, lib.oracle_scatter,
                  lib.oracle_gather, lib.oracle_box_scatter_ids):
            f.restype = None
        _lib = lib
    return _lib


_OMP_SRC = os.path.join(_HERE, "oracle_omp.c")
_OMP_LIB = os.path.join(_HERE, "liboracle_omp.so")
_omp = None


def build_omp(force: bool = False):
    """Compile oracle_omp.c (the oracle's loops on every core, OpenMP) into
    liboracle_omp.so; returns its path, or None when the C compiler has no
    OpenMP."""
    if force or not os.path.exists(_OMP_LIB) or os.path.getmtime(_OMP_LIB) < os.path.getmtime(_OMP_SRC):
        tmp = _OMP_LIB + f".tmp{os.getpid()}"
        res = subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _OMP_SRC, "-lm"],
            capture_output=True,
        )
        if res.returncode != 0:
            return None
        os.replace(tmp, _OMP_LIB)
    return _OMP_LIB


def _load_omp():
    global _omp
    if _omp is None:
        path = build_omp()
        if path is None:
            raise RuntimeError("no OpenMP C compiler: the all-core oracle is not available")
        lib = ctypes.CDLL(path)
        lib.oracle_omp_threads.restype = ctypes.c_int
        lib.oracle_omp_copy.argtypes = [_i64, _f64p, _f64p]
        lib.oracle_omp_axpy.argtypes = [_i64, _dbl, _f64p, _dbl, _f64p, _f64p]
        lib.oracle_omp_dot2.argtypes = [_i64, _f64p, _f64p]
        lib.oracle_omp_dot2.restype = _dbl
        lib.oracle_omp_cg_update.argtypes = [_i64, _dbl, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p]
        lib.oracle_omp_scatter.argtypes = [_i64, _i32p, _f64p, _f64p]
        _i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
        lib.oracle_omp_gather.argtypes = [_i64, _i64, _i64p, _i32p, _f64p, _f64p]
        lib.oracle_rows.argtypes = [_i64, _i64, _i32p, _i64p, _i32p]
        lib.oracle_rows.restype = ctypes.c_int
        for f in (lib.oracle_omp_copy, lib.oracle_omp_axpy, lib.oracle_omp_cg_update,
                  lib.oracle_omp_scatter, lib.oracle_omp_gather):
            f.restype = None
        _omp = lib
    return _omp


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def copy(x):
    """BS1: y = x."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_copy(x.size, x, y)
    return y


def axpy(alpha, x, beta, y):
    """BS2: returns fma(alpha, x_i, beta*y_i) (y is not modified)."""
    x = _f64(x)
    out = np.array(y, dtype=np.float64, copy=True, order="C")
    assert out.size == x.size
    _load().oracle_axpy(x.size, float(alpha), x, float(beta), out)
    return out


def dot(x, y):
    """BS4: Dot2 accurate inner product, summed in index order."""
    x, y = _f64(x), _f64(y)
    assert x.size == y.size
    return float(_load().oracle_dot2(x.size, x, y))


def dot_plain(x, y):
    """Plain sequential inner product (every step rounded)."""
    x, y = _f64(x), _f64(y)
    assert x.size == y.size
    return float(_load().oracle_dot_plain(x.size, x, y))


def norm(x):
    """BS3: x.x (the squared 2-norm), by Dot2."""
    x = _f64(x)
    return float(_load().oracle_dot2(x.size, x, x))


def cg_update(alpha, p, Ap, x, r):
    """BS5: returns (x + alpha p, r - alpha Ap, r_new . r_new); inputs untouched."""
    p, Ap = _f64(p), _f64(Ap)
    xo = np.array(x, dtype=np.float64, copy=True, order="C")
    ro = np.array(r, dtype=np.float64, copy=True, order="C")
    n = p.size
    assert Ap.size == n and xo.size == n and ro.size == n
    lib = _load()
    lib.oracle_cg_update(n, float(alpha), p, Ap, xo, ro)
    return xo, ro, float(lib.oracle_dot2(n, ro, ro))


def scatter(ids, qG):
    """BS7: q_L = Z q_G through the local-to-global table (negative id -> 0)."""
    ids, qG = _i32(ids), _f64(qG)
    qL = np.empty(ids.size, dtype=np.float64)
    _load().oracle_scatter(ids.size, ids, qG, qL)
    return qL


def gather(ids, qL, NG):
    """BS6: q_G = Z^T q_L, each global value summed in ascending local index."""
    ids, qL = _i32(ids), _f64(qL)
    assert ids.size == qL.size
    qG = np.empty(int(NG), dtype=np.float64)
    _load().oracle_gather(ids.size, int(NG), ids, qL, qG)
    return qG


def box_scatter_ids(E, N, elem_perm, node_perm, mask_boundary=False, orient=None):
    """Local-to-global table of an E^3 box mesh of degree N (int32, -1 = masked);
    orient[e] in [0, 24) rotates lattice element e's local numbering."""
    ep, npm = _i32(elem_perm), _i32(node_perm)
    assert ep.size == E ** 3 and npm.size == (E * N + 1) ** 3
    ids = np.empty(E ** 3 * (N + 1) ** 3, dtype=np.int32)
    if orient is not None:
        orient = np.ascontiguousarray(orient, dtype=np.uint8)
        assert orient.size == E ** 3 and int(orient.max(initial=0)) < 24
    _load().oracle_box_scatter_ids(int(E), int(N), ep, npm, int(bool(mask_boundary)),
                                   orient.ctypes.data if orient is not None else None, ids)
    return ids


def apply_diag(ids, dL, xG):
    """y_G = Z^T (d_L .* (Z x_G)): the global operator of a diagonal local
    operator ("Portable high-order finite element kernels I", eqs. (6)-(7)).
    Scatter, one rounded product per local value, gather in ascending local
    order."""
    qL = scatter(ids, xG)
    return gather(ids, _f64(dL) * qL, np.asarray(xG).size)


def _quot(num, den):
    """A CG coefficient num / den, or 0 where den is 0 (reading: a vanishing
    p.Ap or r.r occurs only at an exact solution, where a zero step keeps x;
    the pages do not say)."""
    return float(num) / float(den) if float(den) != 0.0 else 0.0


def cg_sequence(ids, pG, xG, rG, rr):
    """One CG iteration's streaming sequence with the identity local operator.

    p_L = Z p_G; Ap_G = Z^T p_L; pAp = p_G . Ap_G; alpha = rr / pAp;
    x += alpha p, r -= alpha Ap with rr_new = r.r; finally rnorm = r.r.
    Returns a dict of every intermediate.
    """
    pG = _f64(pG)
    pL = scatter(ids, pG)
    ApG = gather(ids, pL, pG.size)
    pAp = dot(pG, ApG)
    alpha = _quot(rr, pAp)
    x1, r1, rr_new = cg_update(alpha, pG, ApG, xG, rG)
    rnorm = norm(r1)
    return dict(pL=pL, ApG=ApG, pAp=pAp, alpha=alpha, x=x1, r=r1, rr_new=rr_new, rnorm=rnorm)


def cg_solve(ids, dL, bG, xG, iters):
    """Conjugate gradients on A = Z^T diag(dL) Z (dL None: A = Z^T Z).

    "Portable high-order finite element kernels I": each benchmark problem
    solves its system by CG (Algorithm 1), whose vector operations are
    y = alpha x + beta y, dot, norm and y = A x, and whose steps 8-10 (the x
    update, the r update and r.r) fuse into BS5.  The listing itself was
    lost; this is the textbook (Hestenes-Stiefel) iteration with exactly
    those operations, in that order:

        r = b - A x  (BS2 with alpha = -1);  p = r;  rr_0 = r.r
        for k < iters:
            Ap = A p;  pAp_k = p.Ap;  alpha = rr_k / pAp_k
            x += alpha p;  r -= alpha Ap;  rr_{k+1} = r.r      (BS5)
            p = r + (rr_{k+1} / rr_k) p                        (BS2, alpha = 1)

    A quotient with a zero denominator is 0 (see _quot).  Returns a dict
    with x, r, p (after the last iteration), rr [iters + 1] and pAp [iters].
    """
    bG = _f64(bG)
    NG = bG.size
    ids = _i32(ids)

    def A(v):
        if dL is None:
            return gather(ids, scatter(ids, v), NG)
        return apply_diag(ids, dL, v)

    x = np.array(xG, dtype=np.float64, copy=True, order="C")
    assert x.size == NG
    r = axpy(-1.0, A(x), 1.0, bG)
    p = copy(r)
    rr = [norm(r)]
    pAp = []
    for k in range(int(iters)):
        Ap = A(p)
        pAp.append(dot(p, Ap))
        x, r, rr_new = cg_update(_quot(rr[k], pAp[k]), p, Ap, x, r)
        rr.append(rr_new)
        p = axpy(1.0, r, _quot(rr_new, rr[k]), p)
    return dict(x=x, r=r, p=p, rr=rr, pAp=pAp)


# ---------------------------------------------------------------------------
# The same loops on every host core (oracle_omp.c), for the bench's all-core
# CPU baseline.  Elementwise operations, scatter and gather are bitwise the
# single-thread oracle's; norm and dot sum each thread's contiguous chunk by
# Dot2 and combine the chunks in order.

def omp_threads():
    """OpenMP threads the all-core loops use."""
    return int(_load_omp().oracle_omp_threads())


def omp_copy(x):
    x = _f64(x)
    y = np.empty_like(x)
    _load_omp().oracle_omp_copy(x.size, x, y)
    return y


def omp_axpy(alpha, x, beta, y):
    x, y = _f64(x), _f64(y)
    assert y.size == x.size
    out = np.empty_like(x)
    _load_omp().oracle_omp_axpy(x.size, float(alpha), x, float(beta), y, out)
    return out


def omp_dot(x, y):
    x, y = _f64(x), _f64(y)
    assert x.size == y.size
    return float(_load_omp().oracle_omp_dot2(x.size, x, y))


def omp_norm(x):
    x = _f64(x)
    return float(_load_omp().oracle_omp_dot2(x.size, x, x))


def omp_cg_update(alpha, p, Ap, x, r):
    p, Ap, x, r = _f64(p), _f64(Ap), _f64(x), _f64(r)
    n = p.size
    assert Ap.size == n and x.size == n and r.size == n
    xo, ro = np.empty_like(p), np.empty_like(p)
    lib = _load_omp()
    lib.oracle_omp_cg_update(n, float(alpha), p, Ap, x, r, xo, ro)
    return xo, ro, float(lib.oracle_omp_dot2(n, ro, ro))


def omp_scatter(ids, qG):
    ids, qG = _i32(ids), _f64(qG)
    qL = np.empty(ids.size, dtype=np.float64)
    _load_omp().oracle_omp_scatter(ids.size, ids, qG, qL)
    return qL


def rows_of(ids, NG):
    """Rows of a local-to-global table (setup, not an operation): rowStarts
    [NG + 1] (int64) and the local ids of each row in ascending order (a
    counting sort in oracle_omp.c)."""
    ids = _i32(ids)
    starts = np.zeros(int(NG) + 1, dtype=np.int64)
    local = np.empty(int(np.count_nonzero(ids >= 0)), dtype=np.int32)
    if _load_omp().oracle_rows(ids.size, int(NG), ids, starts, local) != 0:
        raise MemoryError("oracle_rows: out of memory")
    return starts, local


def omp_gather(rows, qL, NG):
    """BS6 on every core: one global row per iteration, ascending local order
    from +0.0 (rows = rows_of(ids, NG))."""
    starts, local = rows
    qL = _f64(qL)
    qG = np.empty(int(NG), dtype=np.float64)
    _load_omp().oracle_omp_gather(qL.size, int(NG), starts, _i32(local), qL, qG)
    return qG
