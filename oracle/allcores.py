"""The oracle's loops on every host core, timed over one bench step --
TEST INFRASTRUCTURE ONLY: the all-core leg of the bench's CPU baseline, run by
``bench.py`` in a process of its own (no PyTorch or CUDA in it, so that only
this process's OpenMP runtime is loaded).

    python -m oracle.allcores <workload> <seconds> [<scatter ids .npy>]

builds the workload's inputs (``bsinputs``, the same seeds and tags as the
bench's single-thread oracle leg) and the rows of the local-to-global table
(read from the .npy file the bench wrote, else built here; setup, not
timed), then repeats the step -- BS1-BS5 at n = N_L, gather,
scatter, and the CG sequence at n = N_G -- with the OpenMP loops of
``oracle_omp.c`` until ``seconds`` have passed, and prints one JSON line:
wall seconds per step and per operation, and the thread count.
"""

from __future__ import annotations

import json
import sys
import time

import numpy as np

import bsinputs as gen
import oracle


def main(argv):
    cfg = gen.WORKLOADS[argv[0]]
    seconds = float(argv[1]) if len(argv) > 1 else 10.0
    NL, NG, s = cfg.NL, cfg.NG, cfg.seed
    if len(argv) > 2:
        ids = np.load(argv[2])
    else:
        ep, npm = gen.mesh_perms(cfg)
        orient = gen.element_orientations(cfg) if cfg.flags & gen.ROTATE_ELEMS else None
        ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm, bool(cfg.flags & gen.MASK_BOUNDARY),
                                     orient)
    assert ids.size == NL
    rows = oracle.rows_of(ids, NG)
    u = gen.uniform_pm1(s, gen.TAG_U, NL)
    p = gen.uniform_pm1(s, gen.TAG_P, NL)
    Ap = gen.uniform_pm1(s, gen.TAG_AP, NL)
    r = gen.uniform_pm1(s, gen.TAG_R, NL)
    x = gen.uniform_pm1(s, gen.TAG_X, NL)
    qG = gen.uniform_pm1(s, gen.TAG_U + 32, NG)
    pG = gen.uniform_pm1(s, gen.TAG_P + 32, NG)
    xG = gen.uniform_pm1(s, gen.TAG_X + 32, NG)
    rG = gen.uniform_pm1(s, gen.TAG_R + 32, NG)
    times = {}
    clock = time.perf_counter

    def step():
        t = [clock()]

        def mark(name):
            t.append(clock())
            times[name] = times.get(name, 0.0) + t[-1] - t[-2]

        oracle.omp_copy(u)
        mark("copy")
        oracle.omp_axpy(cfg.alpha, p, cfg.beta, r)
        mark("axpy")
        oracle.omp_norm(Ap)
        mark("norm")
        oracle.omp_dot(x, u)
        mark("dot")
        oracle.omp_cg_update(cfg.alpha, p, Ap, x, r)
        mark("cg_update")
        oracle.omp_gather(rows, u, NG)
        mark("gather")
        oracle.omp_scatter(ids, qG)
        mark("scatter")
        pL = oracle.omp_scatter(ids, pG)
        ApG = oracle.omp_gather(rows, pL, NG)
        pAp = oracle.omp_dot(pG, ApG)
        _, r1, _ = oracle.omp_cg_update(1.0 / (pAp or 1.0), pG, ApG, xG, rG)
        oracle.omp_norm(r1)
        mark("cg_iteration")

    step()  # warm-up: first touch of the outputs' pages
    times.clear()
    reps = 0
    t0 = clock()
    while True:
        step()
        reps += 1
        dt = clock() - t0
        if dt >= seconds or reps >= 50:
            break
    print(json.dumps({"workload": cfg.name, "threads": oracle.omp_threads(), "reps": reps,
                      "seconds": dt, "s_per_step": dt / reps,
                      "s_per_op": {k: v / reps for k, v in times.items()}}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
