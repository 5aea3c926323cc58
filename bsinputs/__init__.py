"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the Benchmark Streaming operations: it only
draws random numbers and states the workload shapes.  Both sides of every
parity comparison consume the arrays made here, byte for byte.

Random source: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-based: the i-th
draw (i = 0, 1, ...) of stream (seed, tag) is

    z_i = mix64(key + (i + 1) * GAMMA)   (mod 2^64),
    key = seed XOR (tag * GAMMA mod 2^64),

which is exactly the i-th output of a SplitMix64 generator whose state starts
at `key`.  mix64 is SplitMix64's output function.

Derived values (all exact in binary64 except the Box-Muller transcendental step):
  * uniform on (-1, 1):  k = z >> 11 (53 bits);  u = (k * 2^-52 - 1) + 2^-53.
    Each step is exact, so u = (2k + 1) 2^-53 - 1, never 0, symmetric.
  * uniform on [a, b):    a + (b - a) * (k * 2^-53).
  * standard normal:      Box-Muller on draws 2i, 2i+1:
        u1 = (k_{2i} + 1) 2^-53 in (0, 1],  u2 = k_{2i+1} 2^-53 in [0, 1),
        n_i = sqrt(-2 ln u1) * cos(2 pi u2).
  * random permutation:   the indices 0..n-1 ordered by (z_i, i), i.e. a
    stable argsort of the first n draws.  slot -> item.

The same definitions are restated in C inside the library's seeded mesh
builder; the tests compare the two bit for bit.
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# Stream tags.  One tag per independently drawn quantity of a configuration.
TAG_ELEM_PERM = 1
TAG_NODE_PERM = 2
TAG_U = 3
TAG_P = 4
TAG_AP = 5
TAG_R = 6
TAG_X = 7
TAG_ALPHA = 8
TAG_Y = 9
TAG_ORIENT = 10
# Tags >= 16 are free for extra vectors a caller needs (e.g. one distinct
# buffer per operation in a timed step).
TAG_EXTRA = 16

SEED_BASE = 0xB5EED000

# Mesh flags (same bit values as the C library's BS_MESH_* flags).
SHUFFLE_ELEMS = 1
PERMUTE_GLOBAL = 2
MASK_BOUNDARY = 4
ROTATE_ELEMS = 8


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (reference form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int) -> int:
    return (seed ^ ((tag * GAMMA) & MASK64)) & MASK64


def draws(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    """z_start .. z_{start+n-1} of stream (seed, tag) as uint64."""
    key = np.uint64(stream_key(seed, tag))
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = key + i * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def _uniform_pm1_block(seed, tag, n, start):
    k = (draws(seed, tag, n, start) >> np.uint64(11)).astype(np.float64)
    return (k * 2.0 ** -52 - 1.0) + 2.0 ** -53


def uniform_pm1(seed: int, tag: int, n: int, threads: int = 0) -> np.ndarray:
    """n binary64 values uniform on (-1, 1).

    Large requests are drawn in blocks on a thread pool (numpy releases the
    GIL); the values do not depend on the blocking (counter-based draws).
    """
    block = 1 << 22
    if n <= block:
        return _uniform_pm1_block(seed, tag, n, 0)
    out = np.empty(n, dtype=np.float64)
    starts = range(0, n, block)

    def fill(a):
        b = min(a + block, n)
        out[a:b] = _uniform_pm1_block(seed, tag, b - a, a)

    workers = threads or min(16, os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(fill, starts))
    return out


def uniform_range(seed: int, tag: int, n: int, a: float, b: float) -> np.ndarray:
    k = (draws(seed, tag, n) >> np.uint64(11)).astype(np.float64)
    return a + (b - a) * (k * 2.0 ** -53)


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    z = draws(seed, tag, 2 * n) >> np.uint64(11)
    u1 = (z[0::2].astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = z[1::2].astype(np.float64) * 2.0 ** -53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    """Random permutation of 0..n-1 (int32): indices ordered by (z_i, i)."""
    if n == 0:
        return np.zeros(0, dtype=np.int32)
    keys = draws(seed, tag, n)
    return np.argsort(keys, kind="stable").astype(np.int32)


def integers_dyadic(seed: int, tag: int, n: int, bits: int = 20) -> np.ndarray:
    """Integers in [-2^bits, 2^bits) as binary64; sums of up to 8 are exact."""
    z = draws(seed, tag, n) >> np.uint64(64 - (bits + 1))
    return z.astype(np.float64) - float(1 << bits)


@dataclasses.dataclass(frozen=True)
class MeshConfig:
    """A box mesh of E^3 hexahedra of degree N on [0,1]^3."""

    name: str
    E: int
    N: int
    seed: int
    flags: int = SHUFFLE_ELEMS | PERMUTE_GLOBAL
    alpha: float = 0.37
    beta: float = 1.0

    @property
    def K(self) -> int:
        return self.E ** 3

    @property
    def Np(self) -> int:
        return (self.N + 1) ** 3

    @property
    def NL(self) -> int:
        return self.K * self.Np

    @property
    def NG(self) -> int:
        return (self.E * self.N + 1) ** 3


# The benchmark workloads: four box meshes (tiny, mid, large, stress) and the
# vector-length sweep 2^10 .. 2^27 for the five mesh-free operations; plus
# the stress mesh with Dirichlet-masked boundary nodes and randomly oriented
# elements (an unstructured-like numbering) at the same scale; plus "probe",
# the stress mesh's degree on 48^3 elements: every vector beyond L2 (191 MB
# local, 112 MB global) with a few GB on the device, the size hardware
# counters are captured at.
WORKLOADS = {
    "tiny": MeshConfig("tiny", 8, 3, SEED_BASE + 0),
    "mid": MeshConfig("mid", 20, 7, SEED_BASE + 1),
    "large": MeshConfig("large", 32, 7, SEED_BASE + 3),
    "stress": MeshConfig("stress", 64, 5, SEED_BASE + 4),
    "stress_masked": MeshConfig("stress_masked", 64, 5, SEED_BASE + 5,
                                SHUFFLE_ELEMS | PERMUTE_GLOBAL | MASK_BOUNDARY | ROTATE_ELEMS),
    "probe": MeshConfig("probe", 48, 5, SEED_BASE + 6),
}
SWEEP_SEED = SEED_BASE + 2
SWEEP_LOG2 = tuple(range(10, 28))


def mesh_perms(cfg: MeshConfig):
    """(elemPerm[K], nodePerm[N_G]) for a configuration, honouring its flags.

    elemPerm[s] is the lattice element stored in slot s; nodePerm[L] is the
    global id given to lattice node L.  Identity when the flag is off.
    """
    if cfg.flags & SHUFFLE_ELEMS:
        ep = permutation(cfg.seed, TAG_ELEM_PERM, cfg.K)
    else:
        ep = np.arange(cfg.K, dtype=np.int32)
    if cfg.flags & PERMUTE_GLOBAL:
        npm = permutation(cfg.seed, TAG_NODE_PERM, cfg.NG)
    else:
        npm = np.arange(cfg.NG, dtype=np.int32)
    return ep, npm


def random_scatter_ids(seed: int, tag: int, NL: int, NG: int, masked_per_256: int = 0) -> np.ndarray:
    """An unstructured local-to-global table (int32): local l maps to global
    ((z_l >> 11) mod NG), or -1 (masked) where (z_l & 255) < masked_per_256.
    Row lengths (copies per global node) are then about Poisson(NL / NG)."""
    z = draws(seed, tag, NL)
    ids = ((z >> np.uint64(11)) % np.uint64(max(NG, 1))).astype(np.int64)
    ids[(z & np.uint64(255)) < np.uint64(masked_per_256)] = -1
    return ids.astype(np.int32)


def element_orientations(cfg: MeshConfig) -> np.ndarray:
    """Orientation index in [0, 24) of every lattice element (uint8), drawn
    as ((z_e >> 11) * 24) >> 53 from stream (seed, TAG_ORIENT); zeros when
    the ROTATE_ELEMS flag is off.  (The rotation an index names is part of
    the mesh numbering, implemented by each table builder.)"""
    if not cfg.flags & ROTATE_ELEMS:
        return np.zeros(cfg.K, dtype=np.uint8)
    z = draws(cfg.seed, TAG_ORIENT, cfg.K) >> np.uint64(11)
    with np.errstate(over="ignore"):
        return ((z * np.uint64(24)) >> np.uint64(53)).astype(np.uint8)


def gll_nodes_weights(N: int):
    """Gauss-Lobatto-Legendre nodes and weights on [-1, 1] (degree N, N+1 points):
    the end points and the roots of P_N'; w_i = 2 / (N (N+1) P_N(x_i)^2)."""
    leg = np.polynomial.legendre.Legendre
    if N == 1:
        x = np.array([-1.0, 1.0])
    else:
        x = np.concatenate([[-1.0], np.sort(leg.basis(N).deriv().roots().real), [1.0]])
    w = 2.0 / (N * (N + 1) * leg.basis(N)(x) ** 2)
    return x, w


def mass_diagonal(E: int, N: int) -> np.ndarray:
    """Diagonal GLL mass matrix of every element of an E^3 box mesh of
    [0,1]^3, degree N, in local order (i fastest): w_i w_j w_k (h/2)^3,
    h = 1/E.  An input coefficient array for the diagonal local operator."""
    _, w = gll_nodes_weights(N)
    q = N + 1
    n = np.arange(q ** 3)
    i, j, k = n % q, (n // q) % q, n // (q * q)
    elem = w[i] * w[j] * w[k] * (0.5 / E) ** 3
    return np.tile(elem, E ** 3)


def sweep_vectors(log2n: int):
    """(x, y, alpha) of the sweep point n = 2^log2n: N(0,1) data, alpha ~ U(0.1, 1)."""
    n = 1 << log2n
    x = normal(SWEEP_SEED, TAG_X + 100 * log2n, n)
    y = normal(SWEEP_SEED, TAG_Y + 100 * log2n, n)
    alpha = float(uniform_range(SWEEP_SEED, TAG_ALPHA + 100 * log2n, 1, 0.1, 1.0)[0])
    return x, y, alpha
