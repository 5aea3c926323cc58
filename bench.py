#!/usr/bin/env python3
"""Bench of the seven Benchmark Streaming operations (BS1-BS7) on GB300.

Default run (one JSON line on stdout, rank 0):
  one step = the whole hot path on the stress mesh (64^3 hexahedra, degree
  5: N_L = 56,623,104 local and N_G = 33,076,161 global nodes, element
  order shuffled, global ids permuted): BS1 copy, BS2 AXPY, BS3 norm, BS4
  dot, BS5 fused CG update at length N_L, BS6 gather, BS7 scatter, and one
  CG iteration's streaming sequence (scatter, gather, dot, fused update,
  norm) on global-length vectors.  Every operation works on its own
  buffers, all larger than L2, so no operation reads what the previous one
  left in L2.
  value = algorithmic bytes of the step / device time of the step (GB/s),
  timed with CUDA events on the launching stream over exactly --steps
  steps after --warmup steps.  Per-kernel times come from events between
  the launches; the dominant kernel's figures form the `roofline` object.

Other modes:
  --impl reference   the CPU oracle timed on a bounded sample of the same
                     workload (the reference arm).
  --sweep            BS1-BS5 at n = 2^10 .. 2^27, host-timed launch->sync
                     as the pages time, with the T(B) = T0 + B/Wmax fit.
  --mass-operator    y = Z^T diag(d) Z x, fused against scatter + gather.
  --cg-solve         CG on Z^T diag(d) Z (GLL mass): time per iteration on
                     --config, eager launches against one CUDA-graph replay,
                     and the same on the tiny mesh, where launches dominate.
  --config NAME      another mesh workload (tiny, mid, large, stress).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bsinputs as gen  # noqa: E402

METRIC = "achieved HBM GB/s per BS1–BS7 kernel and fraction of measured GB300 peak"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SRC = {
    "copy": ("bs_vec.cu",), "axpy": ("bs_vec.cu",), "norm": ("bs_vec.cu",), "dot": ("bs_vec.cu",),
    "cg_update": ("bs_vec.cu",), "gather": ("bs_gs.cu", "bs_gs2.cu"),
    "scatter": ("bs_gs.cu", "bs_gs2.cu"),
}
# Library kernels of one default (two-pass) step, in launch order, and the
# operation each belongs to.
STEP_KERNELS = [
    ("copy_kernel", "copy"), ("axpy_kernel", "axpy"), ("dot_kernel", "norm"),
    ("dot_kernel", "dot"), ("cg_kernel", "cg_update"), ("gather_tile_kernel", "gather"),
    ("gather_bucket_tm_kernel", "gather"), ("scatter_tile_kernel", "scatter"),
    ("scatter_bucket_kernel", "scatter"), ("scatter_tile_kernel", "cg_iteration"),
    ("scatter_bucket_kernel", "cg_iteration"), ("gather_tile_kernel", "cg_iteration"),
    ("gather_bucket_tm_kernel", "cg_iteration"), ("dot_kernel", "cg_iteration"),
    ("cg_kernel", "cg_iteration"), ("dot_kernel", "cg_iteration"),
]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", choices=sorted(gen.WORKLOADS), default="stress")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-sample", type=float, default=1.0,
                    help="fraction of the step the oracle runs for cpu_baseline")
    ap.add_argument("--no-all-cores", action="store_true",
                    help="skip the all-core (OpenMP) oracle leg of cpu_baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="repeat the oracle sample until this much CPU time has passed")
    ap.add_argument("--ref-sample", type=float, default=1.0 / 32,
                    help="fraction of the step per reference-arm step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--mass-operator", action="store_true",
                    help="time y = Z^T diag(d) Z x (fused, GLL mass diagonal) against a "
                         "separate scatter + gather on --config")
    ap.add_argument("--cg-solve", action="store_true",
                    help="time CG iterations on the GLL mass operator (eager and CUDA graph)")
    ap.add_argument("--cg-iters", type=int, default=20)
    ap.add_argument("--no-plan", action="store_true",
                    help="one-pass gather/scatter kernels instead of the two-pass plan")
    ap.add_argument("--norm-ab", action="store_true",
                    help="BS3 norm at n = N_L of --config timed after a read-only operation "
                         "and after operations that write N_L values (AXPY, copy)")
    ap.add_argument("--cg-no-compare", action="store_true",
                    help="--cg-solve on --config only (skip the tiny- and mid-mesh comparisons)")
    ap.add_argument("--traffic-from", metavar="CSV", nargs="+",
                    help="write profiles/ncu_traffic.json from per-kernel ncu captures (CSV with "
                         "dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum) "
                         "of one default step on --traffic-capture, scaled to --config, then exit")
    ap.add_argument("--traffic-capture", default="large", choices=sorted(gen.WORKLOADS),
                    help="the mesh the --traffic-from captures ran on")
    ap.add_argument("--soak", type=float, default=1.5,
                    help="seconds of untimed steps before warm-up (clock sampling)")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def src_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "order_fem_cg_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(kernel, config):
    """ncu DRAM bytes per launch of `kernel`, if captured on the current source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)["kernels"][kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("src_sha256") != src_sha(KERNEL_SRC[kernel]) or rec.get("config") != config:
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summary()

    def summary(self):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        rows = [r for r in self.rows if num(r[0]) is not None]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if (num(r[3]) or 0) >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(num(r[0]) for r in loaded),
                "sm_max_mhz": max(num(r[1]) or 0 for r in loaded),
                "power_w_max": max(num(r[2]) or 0 for r in loaded),
                "reasons": reasons, "samples": len(loaded)}


# --------------------------------------------------------------- workload

class Workload:
    """Device buffers and the launch list of one step on a mesh configuration."""

    N_VEC_L = ("a", "b", "c", "d", "e", "f", "g", "P", "AP", "X", "R", "qL1", "qL2", "pL")
    N_VEC_G = ("qG1", "qG2", "pG", "ApG", "xG", "rG")

    def __init__(self, cfg, torch, bs, device, planned=True):
        self.cfg, self.torch, self.bs, self.device = cfg, torch, bs, device
        self.mesh = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
        if self.mesh.validate() != bs.BS_OK:
            raise RuntimeError("mesh tables failed validation")
        self.tables = self.mesh.to_device(device.index, planned=planned)
        self.planned = self.tables.plan is not None
        NL, NG = cfg.NL, cfg.NG
        self.NL, self.NG = NL, NG
        s = cfg.seed
        # host inputs (seeded); several device buffers share values
        self.h = {
            "u": gen.uniform_pm1(s, gen.TAG_U, NL), "p": gen.uniform_pm1(s, gen.TAG_P, NL),
            "Ap": gen.uniform_pm1(s, gen.TAG_AP, NL), "r": gen.uniform_pm1(s, gen.TAG_R, NL),
            "x": gen.uniform_pm1(s, gen.TAG_X, NL),
            "qG": gen.uniform_pm1(s, gen.TAG_U + 32, NG), "pG": gen.uniform_pm1(s, gen.TAG_P + 32, NG),
            "xG": gen.uniform_pm1(s, gen.TAG_X + 32, NG), "rG": gen.uniform_pm1(s, gen.TAG_R + 32, NG),
        }
        self.src = {"a": "u", "c": "p", "d": "r", "e": "Ap", "f": "x", "g": "u", "P": "p",
                    "AP": "Ap", "X": "x", "R": "r", "qL1": "u", "qG2": "qG", "pG": "pG",
                    "xG": "xG", "rG": "rG"}
        self.v = {}
        for k in self.N_VEC_L:
            self.v[k] = torch.empty(NL, dtype=torch.float64, device=device)
        for k in self.N_VEC_G:
            self.v[k] = torch.empty(NG, dtype=torch.float64, device=device)
        for k, src in self.src.items():
            self.v[k].copy_(torch.from_numpy(self.h[src]))
        self.rr_host = float(np.dot(self.h["rG"], self.h["rG"]))
        self.sc = {k: torch.zeros(1, dtype=torch.float64, device=device)
                   for k in ("norm", "dot", "rdotr", "rr", "pAp", "rr_new", "rnorm")}
        self.sc["rr"].fill_(self.rr_host)
        torch.cuda.synchronize()
        pm = bs_perf()
        t = self.tables
        self.bytes = {
            "copy": pm.bytes_copy(NL), "axpy": pm.bytes_axpy(NL), "norm": pm.bytes_norm(NL),
            "dot": pm.bytes_dot(NL), "cg_update": pm.bytes_cg_update(NL),
            "gather": pm.bytes_gather(NL, NG, t.nnz, t.nblocks),
            "scatter": pm.bytes_scatter(NL, NG),
            "cg_iteration": pm.bytes_cg_iteration(NL, NG, t.nnz, t.nblocks),
        }
        g_l, s_l = bs.gs_launches(cfg.NL, cfg.NG, self.planned)
        self.launches = {"copy": 1, "axpy": 1, "norm": 1, "dot": 1, "cg_update": 1, "gather": g_l,
                         "scatter": s_l, "cg_iteration": 3 + g_l + s_l}
        self.names = list(self.bytes)

    @property
    def step_bytes(self):
        return sum(self.bytes.values())

    @property
    def launches_per_step(self):
        return sum(self.launches.values())

    def op(self, name, stream):
        bs, v, sc, cfg = self.bs, self.v, self.sc, self.cfg
        if name == "copy":
            bs.bs_copy(v["a"], v["b"], stream)
        elif name == "axpy":
            bs.bs_axpy(cfg.alpha, v["c"], cfg.beta, v["d"], stream)
        elif name == "norm":
            bs.bs_norm(v["e"], sc["norm"], stream)
        elif name == "dot":
            bs.bs_dot(v["f"], v["g"], sc["dot"], stream)
        elif name == "cg_update":
            bs.bs_cg_update(v["P"], v["AP"], v["X"], v["R"], alpha=cfg.alpha, rdotr=sc["rdotr"],
                            stream=stream)
        elif name == "gather":
            bs.bs_gather(self.tables, v["qL1"], v["qG1"], stream)
        elif name == "scatter":
            bs.bs_scatter(self.tables, v["qG2"], v["qL2"], stream)
        elif name == "cg_iteration":
            bs.bs_cg_iteration(self.tables, v["pG"], v["pL"], v["ApG"], v["xG"], v["rG"], sc["rr"],
                               sc["pAp"], sc["rr_new"], sc["rnorm"], stream)
        else:
            raise KeyError(name)

    def step(self, stream, events=None):
        for i, name in enumerate(self.names):
            self.op(name, stream)
            if events is not None:
                events[i + 1].record(stream)

    # -- end to end: host buffers in, host buffers out
    INPUTS = ("a", "c", "d", "e", "f", "g", "P", "AP", "X", "R", "qL1", "qG2", "pG", "xG", "rG")
    OUTPUTS = ("b", "d", "X", "R", "qG1", "qL2", "xG", "rG")

    def pin_host(self):
        torch = self.torch
        self.hin = {k: torch.from_numpy(self.h[self.src[k]]).pin_memory() for k in self.INPUTS}
        self.hout = {k: torch.empty(self.v[k].numel(), dtype=torch.float64).pin_memory()
                     for k in self.OUTPUTS}
        self.hsc_in = torch.tensor([self.rr_host], dtype=torch.float64).pin_memory()
        self.hsc_out = torch.empty(len(self.sc), dtype=torch.float64).pin_memory()
        self.sc_cat = torch.empty(len(self.sc), dtype=torch.float64, device=self.device)

    @property
    def h2d_bytes(self):
        return sum(t.numel() * 8 for t in self.hin.values()) + 8

    @property
    def d2h_bytes(self):
        return sum(t.numel() * 8 for t in self.hout.values()) + 8 * len(self.sc)

    # inputs and outputs of every operation, for the pipelined end-to-end step
    OP_IO = {
        "copy": (("a",), ("b",)), "axpy": (("c", "d"), ("d",)), "norm": (("e",), ()),
        "dot": (("f", "g"), ()), "cg_update": (("P", "AP", "X", "R"), ("X", "R")),
        "gather": (("qL1",), ("qG1",)), "scatter": (("qG2",), ("qL2",)),
        "cg_iteration": (("pG", "xG", "rG"), ("xG", "rG")),
    }

    def e2e_setup(self, compute_stream):
        """Streams and events of the pipelined end-to-end step: each operation's
        inputs go in on a copy-in stream, its kernels run on the compute stream
        once they have landed, its outputs go out on a copy-out stream, so the
        copies of one operation overlap the kernels of its neighbours."""
        torch = self.torch
        self.s_in = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self.s_comp = compute_stream
        mk = lambda: {n: torch.cuda.Event() for n in self.names}  # noqa: E731
        self.ev_in, self.ev_done, self.ev_out = mk(), mk(), mk()
        self.ev_scalars_out = torch.cuda.Event()
        torch.cuda.synchronize()
        for n in self.names:            # first step: nothing to wait for
            self.ev_out[n].record(self.s_out)
        self.ev_scalars_out.record(self.s_out)

    def step_e2e(self):
        torch = self.torch
        # the reductions below overwrite the scalars the previous step reads back
        self.s_comp.wait_event(self.ev_scalars_out)
        for n in self.names:
            ins, outs = self.OP_IO[n]
            with torch.cuda.stream(self.s_in):
                # the previous step's kernels and copy-out of this operation are done
                self.s_in.wait_event(self.ev_out[n])
                for k in ins:
                    self.v[k].copy_(self.hin[k], non_blocking=True)
                if n == "cg_iteration":
                    self.s_in.wait_event(self.ev_scalars_out)
                    self.sc["rr"].copy_(self.hsc_in, non_blocking=True)
                self.ev_in[n].record(self.s_in)
            self.s_comp.wait_event(self.ev_in[n])
            self.op(n, self.s_comp)
            self.ev_done[n].record(self.s_comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(self.ev_done[n])
                for k in outs:
                    self.hout[k].copy_(self.v[k], non_blocking=True)
                self.ev_out[n].record(self.s_out)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_done[self.names[-1]])
            torch.cat([self.sc[k] for k in self.sc], out=self.sc_cat)
            self.hsc_out.copy_(self.sc_cat, non_blocking=True)
            self.ev_scalars_out.record(self.s_out)


_PERFMODEL = None


def bs_perf():
    """order_fem_cg_gb300/perfmodel.py (byte counts, eqs. (8)-(10)) loaded by
    path: importing the package would map libbs.so, and the reference arm
    runs the oracle alone."""
    global _PERFMODEL
    if _PERFMODEL is None:
        import importlib.util
        path = os.path.join(ROOT, "order_fem_cg_gb300", "perfmodel.py")
        spec = importlib.util.spec_from_file_location("_bs_perfmodel", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        _PERFMODEL = mod
    return _PERFMODEL


def host_cpu():
    """The host's logical CPU count and model name (the CPU legs' context)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}


# --------------------------------------------------------- oracle (CPU) leg

class OracleSample:
    """The oracle on a bounded sample of the step: every operation on the
    first `frac` of its local-length range (the CG sequence on the first
    `frac` of its global-length vectors and local entries)."""

    def __init__(self, cfg, frac, host=None):
        import oracle
        self.oracle = oracle
        self.cfg = cfg
        ep, npm = gen.mesh_perms(cfg)
        orient = gen.element_orientations(cfg) if cfg.flags & gen.ROTATE_ELEMS else None
        self.ids = oracle.box_scatter_ids(cfg.E, cfg.N, ep, npm, bool(cfg.flags & gen.MASK_BOUNDARY),
                                          orient)
        NL, NG = cfg.NL, cfg.NG
        self.m = max(1, int(NL * frac))
        self.mg = max(1, int(NG * frac))
        self.frac = frac
        s = cfg.seed
        h = host or {}
        self.u = h.get("u", gen.uniform_pm1(s, gen.TAG_U, NL))[: self.m]
        self.p = h.get("p", gen.uniform_pm1(s, gen.TAG_P, NL))[: self.m]
        self.Ap = h.get("Ap", gen.uniform_pm1(s, gen.TAG_AP, NL))[: self.m]
        self.r = h.get("r", gen.uniform_pm1(s, gen.TAG_R, NL))[: self.m]
        self.x = h.get("x", gen.uniform_pm1(s, gen.TAG_X, NL))[: self.m]
        self.qG = h.get("qG", gen.uniform_pm1(s, gen.TAG_U + 32, NG))
        self.pG = h.get("pG", gen.uniform_pm1(s, gen.TAG_P + 32, NG))
        self.xG = h.get("xG", gen.uniform_pm1(s, gen.TAG_X + 32, NG))
        self.rG = h.get("rG", gen.uniform_pm1(s, gen.TAG_R + 32, NG))
        pm = bs_perf()
        # the full step's algorithmic bytes (blockStarts omitted: negligible)
        full = (pm.bytes_copy(NL) + pm.bytes_axpy(NL) + pm.bytes_norm(NL) + pm.bytes_dot(NL)
                + pm.bytes_cg_update(NL) + pm.bytes_gather(NL, NG, NL, 0) + pm.bytes_scatter(NL, NG)
                + pm.bytes_cg_iteration(NL, NG, NL, 0))
        self.bytes = frac * full

    def step(self, times=None):
        """One sampled step; with `times` (a dict), adds each operation's
        wall time to it."""
        o, cfg, m, mg = self.oracle, self.cfg, self.m, self.mg
        clock = time.perf_counter
        t = [clock()]

        def mark(name):
            t.append(clock())
            if times is not None:
                times[name] = times.get(name, 0.0) + t[-1] - t[-2]

        o.copy(self.u)
        mark("copy")
        o.axpy(cfg.alpha, self.p, cfg.beta, self.r)
        mark("axpy")
        o.norm(self.Ap)
        mark("norm")
        o.dot(self.x, self.u)
        mark("dot")
        o.cg_update(cfg.alpha, self.p, self.Ap, self.x, self.r)
        mark("cg_update")
        o.gather(self.ids[:m], self.u, cfg.NG)
        mark("gather")
        o.scatter(self.ids[:m], self.qG)
        mark("scatter")
        # CG sequence on the sample: scatter/gather over m local entries,
        # vector operations over the first mg global entries
        pL = o.scatter(self.ids[:m], self.pG)
        ApG = o.gather(self.ids[:m], pL, cfg.NG)
        pAp = o.dot(self.pG[:mg], ApG[:mg])
        _, r1, _ = o.cg_update(1.0 / (pAp or 1.0), self.pG[:mg], ApG[:mg], self.xG[:mg],
                               self.rG[:mg])
        o.norm(r1)
        mark("cg_iteration")

    def per_op(self, times, reps):
        """Per-operation oracle figures from accumulated step times: seconds
        per full (unsampled) call and GB/s of the operation's sampled
        algorithmic bytes."""
        pm = bs_perf()
        cfg, f = self.cfg, self.frac
        NL, NG = cfg.NL, cfg.NG
        full = {"copy": pm.bytes_copy(NL), "axpy": pm.bytes_axpy(NL), "norm": pm.bytes_norm(NL),
                "dot": pm.bytes_dot(NL), "cg_update": pm.bytes_cg_update(NL),
                "gather": pm.bytes_gather(NL, NG, NL, 0), "scatter": pm.bytes_scatter(NL, NG),
                "cg_iteration": pm.bytes_cg_iteration(NL, NG, NL, 0)}
        out = {}
        for k, sec in times.items():
            per_call = sec / reps
            out[k] = {"ms_per_full_call": per_call / f * 1e3,
                      "GB/s": f * full[k] / per_call / 1e9}
        return out

    def describe(self):
        return (f"oracle (single-threaded C, Dot2 reductions) on {self.frac:.4g} of the step: "
                f"BS1-BS5 on the first {self.m} of {self.cfg.NL} entries, gather/scatter over the "
                f"first {self.m} local entries, the CG sequence on the first {self.mg} of "
                f"{self.cfg.NG} global entries; GB/s = sampled algorithmic bytes / wall time")


def all_cores_baseline(cfg, seconds, ids=None):
    """The oracle's loops on every host core (oracle/oracle_omp.c, OpenMP:
    elementwise operations, scatter and gather bitwise the single-thread
    oracle's; norm and dot by Dot2 per thread chunk, chunks combined in
    order), run in a process of its own -- no PyTorch, so only one OpenMP
    runtime -- over the full step for `seconds`.  A run that fails is
    reported, not raised."""
    import tempfile
    cmd = [sys.executable, "-m", "oracle.allcores", cfg.name, str(seconds)]
    with tempfile.TemporaryDirectory() as tmp:
        if ids is not None:  # the table the single-thread leg built (saves rebuilding it)
            path = os.path.join(tmp, "ids.npy")
            np.save(path, np.ascontiguousarray(ids, dtype=np.int32))
            cmd.append(path)
        try:
            res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True,
                                 timeout=3 * seconds + 180)
        except subprocess.TimeoutExpired:
            return {"unavailable": "the all-core oracle run did not finish in time"}
    lines = res.stdout.strip().splitlines()
    if res.returncode != 0 or not lines:
        why = (res.stderr.strip().splitlines() or ["no output"])[-1]
        return {"unavailable": f"the all-core oracle run failed: {why[:200]}"}
    d = json.loads(lines[-1])
    pm = bs_perf()
    NL, NG = cfg.NL, cfg.NG
    full = {"copy": pm.bytes_copy(NL), "axpy": pm.bytes_axpy(NL), "norm": pm.bytes_norm(NL),
            "dot": pm.bytes_dot(NL), "cg_update": pm.bytes_cg_update(NL),
            "gather": pm.bytes_gather(NL, NG, NL, 0), "scatter": pm.bytes_scatter(NL, NG),
            "cg_iteration": pm.bytes_cg_iteration(NL, NG, NL, 0)}
    step_bytes = sum(full.values())
    return {"value": step_bytes / d["s_per_step"] / 1e9, "unit": "GB/s", "cores": d["threads"],
            "kind": "oracle loops on all host cores (OpenMP)",
            "reductions": "Dot2 over each thread's contiguous chunk, chunks combined in order",
            "sample": f"{d['reps']} x the full step", "seconds": d["seconds"],
            "per_op": {k: {"ms_per_full_call": v * 1e3, "GB/s": full[k] / v / 1e9}
                       for k, v in d["s_per_op"].items()}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = gen.WORKLOADS[args.config]
    samp = OracleSample(cfg, args.ref_sample)
    for _ in range(args.warmup):
        samp.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        samp.step()
    dt = time.perf_counter() - t0
    value = samp.bytes * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(cfg, args.gpus),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": samp.describe(), "host": host_cpu()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def mesh_numbering(cfg):
    """Plain words for a mesh workload's numbering flags."""
    parts = [("elements shuffled", gen.SHUFFLE_ELEMS), ("global ids permuted", gen.PERMUTE_GLOBAL),
             ("elements randomly oriented", gen.ROTATE_ELEMS),
             ("boundary nodes masked (Dirichlet)", gen.MASK_BOUNDARY)]
    on = [w for w, f in parts if cfg.flags & f]
    return ", ".join(on) if on else "lattice numbering"


def workload_config(cfg, gpus, planned=None):
    out = {
        "workload": f"{cfg.name} box mesh E={cfg.E} N={cfg.N}: {cfg.K} hexahedra, N_L={cfg.NL} local "
                    f"and N_G={cfg.NG} global nodes, {mesh_numbering(cfg)} by "
                    f"seed {cfg.seed:#x}; fp64 U(-1,1) data, alpha={cfg.alpha}, beta={cfg.beta}; step = "
                    "BS1-BS5 at n=N_L, BS6 gather, BS7 scatter, one CG iteration's sequence at n=N_G",
        "l2": (f"inputs larger than L2: every operation streams its own buffers of >= "
               f"{8 * cfg.NG / 1e6:.0f} MB (L2 is 129 MB)" if 8 * cfg.NG > 129e6 else
               f"inputs NOT larger than L2 ({8 * cfg.NL / 1e6:.1f} MB per local vector, L2 129 MB): "
               "figures include L2 reuse"),
        "parallelism": f"replicas x{gpus} (independent meshes, no collective)",
    }
    if planned is not None:
        out["gather_scatter"] = ("two-pass tiled (shared-memory permutation, runs in HBM)"
                                 if planned else "one-pass (random 8-byte accesses)")
    return out


# ------------------------------------------------------------ GPU leg

def aggregate_ranks(dist, torch, elapsed_ms, units, steps, device=None):
    """Whole-job timing over ranks: the slowest rank's time, and the bytes all
    ranks processed per second (weak scaling: every rank runs its own mesh).
    Returns (max elapsed ms, world size, GB/s)."""
    world = 1
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return elapsed_ms, world, units * world * steps / (elapsed_ms * 1e-3) / 1e9


def init_dist(torch, world, local_rank):
    if world <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend, device_id=torch.device("cuda", local_rank)
                            if backend == "nccl" else None)
    return dist


def run_gpu(args):
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = init_dist(torch, world, local_rank)
    import order_fem_cg_gb300 as bs

    cfg = gen.WORKLOADS[args.config]
    wl = Workload(cfg, torch, bs, device, planned=not args.no_plan)
    stream = torch.cuda.Stream(device)
    peak, peak_src = measured_peak()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    # untimed soak so that the clock samples see this load, then warm-up
    t_end = time.perf_counter() + args.soak
    while time.perf_counter() < t_end:
        wl.step(stream)
        stream.synchronize()
    for _ in range(args.warmup):
        wl.step(stream)
    stream.synchronize()

    nops = len(wl.names)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier()
    start.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        wl.step(stream, ev[k])
    stop.record(stream)
    stop.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed_ms, world, value = aggregate_ranks(dist, torch, start.elapsed_time(stop),
                                               wl.step_bytes, args.steps, device)
    ms_per_step = elapsed_ms / args.steps

    per = {}
    for i, name in enumerate(wl.names):
        ms = [ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)]
        avg = sum(ms) / len(ms)
        gbs = wl.bytes[name] / (avg * 1e-3) / 1e9
        per[name] = {"ms": avg, "ms_min": min(ms), "bytes": wl.bytes[name], "GB/s": gbs,
                     "frac": gbs / peak, "launches": wl.launches[name]}
    single = [n for n in per if n != "cg_iteration"]
    dom = max(single, key=lambda n: per[n]["ms"])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": per[dom]["GB/s"], "peak": peak,
                "unit": "GB/s", "frac": per[dom]["GB/s"] / peak,
                "traffic": ncu_traffic(dom, cfg.name),
                "algorithmic_bytes": wl.bytes[dom], "peak_source": peak_src,
                "launches": wl.launches[dom]}

    e2e = None
    if not args.no_e2e:
        wl.pin_host()
        wl.e2e_setup(stream)
        n_e = max(1, min(args.e2e_steps, args.steps))
        wl.step_e2e()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(wl.s_in)
        for _ in range(n_e):
            wl.step_e2e()
        wl.s_out.wait_event(wl.ev_done[wl.names[-1]])
        e1.record(wl.s_out)
        e1.synchronize()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier()
        e_ms = e0.elapsed_time(e1)
        e2e = {"value": wl.step_bytes * world * n_e / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": wl.h2d_bytes, "d2h_bytes_per_step": wl.d2h_bytes,
               "steps": n_e, "ms_per_step": e_ms / n_e, "host_wall_ms_per_step": wall * 1e3 / n_e,
               "pipeline": "per operation: copy-in stream -> compute stream -> copy-out stream"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        samp = OracleSample(cfg, args.cpu_sample, host=wl.h)
        reps = 0
        op_times = {}
        t0 = time.perf_counter()
        while True:
            samp.step(op_times)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= args.cpu_seconds or reps >= 50:
                break
        cpu = {"value": samp.bytes * reps / dt / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{reps} x " + samp.describe(), "seconds": dt,
               "host": host_cpu(), "per_op": samp.per_op(op_times, reps)}
        if not args.no_all_cores:
            cpu["all_cores"] = all_cores_baseline(cfg, args.cpu_seconds, samp.ids)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, world, wl.planned), "roofline": roofline, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": wl.launches_per_step * args.steps, "clocks": clocks,
            "kernels": per, "step_bytes": wl.step_bytes,
            "peak": {"hbm_gbs": peak, "source": peak_src},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ sweep

def run_sweep(args):
    import torch

    import order_fem_cg_gb300 as bs
    from order_fem_cg_gb300 import perfmodel as pm

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peak, peak_src = measured_peak()
    ops = {
        "copy": (pm.bytes_copy, lambda v, a: bs.bs_copy(v[0], v[1])),
        "axpy": (pm.bytes_axpy, lambda v, a: bs.bs_axpy(a, v[0], 1.0, v[1])),
        "norm": (pm.bytes_norm, lambda v, a: bs.bs_norm(v[0], v[4])),
        "dot": (pm.bytes_dot, lambda v, a: bs.bs_dot(v[0], v[1], v[4])),
        "cg_update": (pm.bytes_cg_update,
                      lambda v, a: bs.bs_cg_update(v[0], v[1], v[2], v[3], alpha=a, rdotr=v[4])),
    }
    res = {k: [] for k in ops}
    cap = torch.cuda.Stream()
    for log2n in gen.SWEEP_LOG2:
        x, y, alpha = gen.sweep_vectors(log2n)
        n = x.size
        v = [torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev),
             torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev),
             torch.zeros(1, dtype=torch.float64, device=dev)]
        reps = 50 if n <= (1 << 20) else 10
        K = 100 if n <= (1 << 20) else 10     # launches per stream / graph sample
        for name, (nbytes, fn) in ops.items():
            for _ in range(3):
                fn(v, alpha)
            torch.cuda.synchronize()
            host_t, dev_t = [], []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0 = time.perf_counter()
                e0.record(stream)
                fn(v, alpha)
                e1.record(stream)
                torch.cuda.synchronize()
                host_t.append(time.perf_counter() - t0)
                dev_t.append(e0.elapsed_time(e1) * 1e-3)
            # K back-to-back launches on one stream, device-timed (no host sync
            # between them): what a pipelined solver pays per operation
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(K):
                fn(v, alpha)
            e1.record(stream)
            e1.synchronize()
            stream_t = e0.elapsed_time(e1) * 1e-3 / K
            # the same K launches replayed from one CUDA graph
            cap.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for _ in range(K):
                    fn(v, alpha)
            g.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            graph_t = e0.elapsed_time(e1) * 1e-3 / K
            del g
            res[name].append((n, nbytes(n), statistics.median(host_t), statistics.median(dev_t),
                              stream_t, graph_t))
        del v
    for name, pts in res.items():
        B = np.array([p[1] for p in pts], dtype=np.float64)
        fits = {}
        for key, col in (("host", 2), ("stream", 4), ("graph", 5)):
            T0, Wmax = pm.fit(B, np.array([p[col] for p in pts]))
            fits[key] = {"T0_us": T0 * 1e6, "Wmax_GBs": Wmax / 1e9, "B08_bytes": pm.b_08(T0, Wmax),
                         "Wmax_frac": Wmax / 1e9 / peak}
        h = fits["host"]
        line = {"mode": "sweep", "op": name, "timer": "host (launch -> synchronize), median",
                "T0_us": h["T0_us"], "Wmax_GBs": h["Wmax_GBs"], "B08_bytes": h["B08_bytes"],
                "Wmax_frac": h["Wmax_frac"], "peak_GBs": peak, "peak_source": peak_src,
                "launch_modes": {
                    "host": "one launch then cudaStreamSynchronize, host clock (the pages' method)",
                    "stream": "back-to-back launches on one stream, CUDA events, per launch",
                    "graph": "the same launches replayed from one CUDA graph, CUDA events"},
                "fits": fits,
                "points": [{"n": p[0], "bytes": p[1], "host_us": p[2] * 1e6, "event_us": p[3] * 1e6,
                            "stream_us": p[4] * 1e6, "graph_us": p[5] * 1e6,
                            "GB/s_host": p[1] / p[2] / 1e9, "GB/s_event": p[1] / p[3] / 1e9}
                           for p in pts]}
        print(json.dumps(line), flush=True)
    return 0


def run_norm_ab(args):
    """BS3 inside a sequence: the norm of its own vector timed (CUDA events
    around it alone) right after another operation on other vectors.  A
    preceding operation that wrote N_L values leaves up to L2's worth of
    dirty lines, which HBM writes back while the norm reads."""
    import torch

    import order_fem_cg_gb300 as bs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cfg = gen.WORKLOADS[args.config]
    n = cfg.NL

    def vec(tag):
        return torch.from_numpy(gen.uniform_pm1(cfg.seed, tag, n)).to(dev)

    x, y, z, w = vec(1), vec(2), vec(3), vec(4)
    out = torch.empty(1, dtype=torch.float64, device=dev)
    s = torch.cuda.current_stream()
    peak, src = measured_peak()
    cases = {"after_dot": lambda: bs.bs_dot(x, y),
             "after_norm": lambda: bs.bs_norm(w),
             "after_axpy": lambda: bs.bs_axpy(0.37, x, 1.0, y),
             "after_copy": lambda: bs.bs_copy(x, y)}
    res = {}
    for name, pre in cases.items():
        ts = []
        for i in range(max(3, args.warmup) + max(5, min(args.steps, 50))):
            pre()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            bs.bs_norm(z, out)
            e1.record(s)
            e1.synchronize()
            if i >= max(3, args.warmup):
                ts.append(e0.elapsed_time(e1) * 1e3)
        med = statistics.median(ts)
        res[name] = {"median_us": med, "min_us": min(ts),
                     "GB/s": 8 * n / (med * 1e-6) / 1e9, "frac": 8 * n / (med * 1e-6) / 1e9 / peak}
    print(json.dumps({"mode": "norm_ab", "workload": cfg.name, "n": n, "peak_source": src,
                      "cases": res}), flush=True)
    return 0


def run_mass_operator(args):
    import torch

    import order_fem_cg_gb300 as bs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cfg = gen.WORKLOADS[args.config]
    mesh = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    t = mesh.to_device(0)
    x = torch.from_numpy(gen.uniform_pm1(cfg.seed, gen.TAG_X, cfg.NG)).to(dev)
    d = torch.from_numpy(gen.mass_diagonal(cfg.E, cfg.N)).to(dev)
    y = torch.empty(cfg.NG, dtype=torch.float64, device=dev)
    qL = torch.empty(cfg.NL, dtype=torch.float64, device=dev)

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    fused = timed(lambda: bs.bs_apply_diag(t, x, d, y), args.steps)
    separate = timed(lambda: (bs.bs_scatter(t, x, qL), bs.bs_gather(t, qL, y)), args.steps)
    # the same arithmetic unfused: scatter, the elementwise product (torch's
    # kernel, one binary64 multiply per local), gather
    unfused = timed(lambda: (bs.bs_scatter(t, x, qL), qL.mul_(d), bs.bs_gather(t, qL, y)),
                    args.steps)
    nbytes = 16 * cfg.NG + 12 * cfg.NL   # read x, d, ids; write y
    peak, src = measured_peak()
    print(json.dumps({"mode": "mass_operator", "workload": cfg.name, "op": "y = Z^T diag(d) Z x",
                      "fused_ms": fused, "scatter_plus_gather_ms": separate,
                      "scatter_times_d_gather_ms": unfused,
                      "algorithmic_bytes": nbytes, "fused_GB/s": nbytes / (fused * 1e-3) / 1e9,
                      "fused_frac": nbytes / (fused * 1e-3) / 1e9 / peak, "peak_source": src,
                      "steps": args.steps}), flush=True)
    return 0


def cg_solve_times(cfg, iters, reps, warmup, torch, bs, dev):
    """(eager ms, graph ms) per CG iteration on cfg's mesh, mass operator:
    a solve of `iters` iterations minus one of 0 iterations (the setup),
    each timed with events over `reps` calls after `warmup` calls."""
    mesh = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    t = mesh.to_device(0)
    NG = cfg.NG
    d = torch.from_numpy(gen.mass_diagonal(cfg.E, cfg.N)).to(dev)
    b = torch.from_numpy(gen.uniform_pm1(cfg.seed, gen.TAG_R, NG)).to(dev)
    x, r, p, Ap = (torch.zeros(NG, dtype=torch.float64, device=dev) for _ in range(4))
    scal = {k: torch.zeros(2 * k + 1, dtype=torch.float64, device=dev) for k in (0, iters)}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def solve(k):
        x.zero_()
        bs.bs_cg_solve(t, d, b, x, r, p, Ap, k, scal[k], stream=s)

    def timed(fn):
        with torch.cuda.stream(s):
            for _ in range(warmup):
                fn()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(reps):
                fn()
            e1.record(s)
            e1.synchronize()
        return e0.elapsed_time(e1) / reps

    eager = {k: timed(lambda k=k: solve(k)) for k in (0, iters)}
    graphs = {}
    for k in (0, iters):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            solve(k)
        graphs[k] = g
    graph = {k: timed(graphs[k].replay) for k in (0, iters)}
    rr = scal[iters].cpu().numpy()[:iters + 1]
    return ((eager[iters] - eager[0]) / iters, (graph[iters] - graph[0]) / iters,
            float(rr[-1] / rr[0]))


def cg_fused_times(cfg, iters, reps, warmup, torch, bs, dev):
    """ms per CG iteration of the one-kernel solve (grid barriers), mass
    operator: a solve of `iters` iterations minus one of 0 iterations."""
    mesh = bs.Mesh(cfg.E, cfg.N, cfg.seed, cfg.flags)
    t = mesh.to_device(0, planned=False)
    NG = cfg.NG
    d = torch.from_numpy(gen.mass_diagonal(cfg.E, cfg.N)).to(dev)
    b = torch.from_numpy(gen.uniform_pm1(cfg.seed, gen.TAG_R, NG)).to(dev)
    x, r, p, Ap = (torch.zeros(NG, dtype=torch.float64, device=dev) for _ in range(4))
    pL = torch.zeros(cfg.NL, dtype=torch.float64, device=dev)
    scal = {k: torch.zeros(2 * k + 1, dtype=torch.float64, device=dev) for k in (0, iters)}

    def timed(k):
        for _ in range(warmup):
            bs.bs_cg_solve_fused(t, d, b, x, r, p, Ap, pL, k, scal[k])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            bs.bs_cg_solve_fused(t, d, b, x, r, p, Ap, pL, k, scal[k])
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    ms = (timed(iters) - timed(0)) / iters
    if bs.default_context().device_status() != bs.BS_OK:
        raise RuntimeError("fused CG solve reported a device error")
    return ms


def run_cg_solve(args):
    import torch

    import order_fem_cg_gb300 as bs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cfg = gen.WORKLOADS[args.config]
    K = max(1, args.cg_iters)
    reps = max(3, min(args.steps, 20))
    eager, graph, rr_ratio = cg_solve_times(cfg, K, reps, max(3, args.warmup), torch, bs, dev)
    # per iteration: y = A p (x, y, d, one index per local), p.Ap, BS5, p update
    nbytes = 16 * cfg.NG + 12 * cfg.NL + 16 * cfg.NG + 48 * cfg.NG + 24 * cfg.NG
    peak, src = measured_peak()
    if args.cg_no_compare:
        print(json.dumps({
            "mode": "cg_solve", "workload": cfg.name, "operator": "A = Z^T diag(GLL mass) Z",
            "iters": K, "rr_ratio": rr_ratio, "eager_ms_per_iter": eager,
            "graph_ms_per_iter": graph, "bytes_per_iter": nbytes,
            "GB/s": nbytes / (graph * 1e-3) / 1e9, "frac": nbytes / (graph * 1e-3) / 1e9 / peak,
            "peak_source": src}), flush=True)
        return 0
    tiny = gen.WORKLOADS["tiny"]
    t_eager, t_graph, _ = cg_solve_times(tiny, 50, 20, 3, torch, bs, dev)
    t_fused = cg_fused_times(tiny, 50, 20, 3, torch, bs, dev)
    mid = gen.WORKLOADS["mid"]
    m_eager, m_graph, _ = cg_solve_times(mid, 20, 10, 3, torch, bs, dev)
    m_fused = cg_fused_times(mid, 20, 10, 3, torch, bs, dev)
    print(json.dumps({
        "mode": "cg_solve", "workload": cfg.name, "operator": "A = Z^T diag(GLL mass) Z",
        "iters": K, "rr_ratio": rr_ratio, "launches_per_iter": 6,
        "eager_ms_per_iter": eager, "graph_ms_per_iter": graph,
        "bytes_per_iter": nbytes, "GB/s": nbytes / (graph * 1e-3) / 1e9,
        "frac": nbytes / (graph * 1e-3) / 1e9 / peak, "peak_source": src,
        "tiny": {"workload": tiny.name, "eager_us_per_iter": 1e3 * t_eager,
                 "graph_us_per_iter": 1e3 * t_graph,
                 "one_kernel_us_per_iter": 1e3 * t_fused,
                 "launch_us_saved_per_kernel": 1e3 * (t_eager - t_graph) / 6},
        "mid": {"workload": mid.name, "eager_us_per_iter": 1e3 * m_eager,
                "graph_us_per_iter": 1e3 * m_graph, "one_kernel_us_per_iter": 1e3 * m_fused}}),
        flush=True)
    return 0


def _ncu_launches(path):
    """{kernel: [(ID, dram bytes, ns), ...] in launch order} of an ncu --csv log."""
    import csv
    import io
    import re
    lines = open(path).read().splitlines()
    head = next(i for i, l in enumerate(lines) if l.startswith('"ID"'))
    launches = {}
    for r in csv.DictReader(io.StringIO("\n".join(lines[head:]))):
        m = re.search(r"<unnamed>::(\w+_kernel)", r["Kernel Name"])
        if not m:
            continue
        rec = launches.setdefault(int(r["ID"]), {"kernel": m.group(1)})
        rec[r["Metric Name"]] = float(r["Metric Value"].replace(",", ""))
    out = {}
    for i in sorted(launches):
        k = launches[i]
        out.setdefault(k["kernel"], []).append(
            (i, k.get("dram__bytes_read.sum", 0.0) + k.get("dram__bytes_write.sum", 0.0),
             k.get("gpu__time_duration.sum", 0.0)))
    return out


def traffic_from_csv(paths, capture, target):
    """Per-operation DRAM bytes per call from per-kernel ncu captures of one
    bench step on the `capture` mesh (each log one kernel family, its first
    launches in step order), scaled to the `target` mesh by the operation's
    moved-bytes model (perfmodel.moved_bytes)."""
    per_kernel = {}
    for p in paths:
        for k, v in _ncu_launches(p).items():
            per_kernel.setdefault(k, []).extend(v)
    used = {}
    ops = {}
    for kernel, op in STEP_KERNELS:
        i = used.get(kernel, 0)
        used[kernel] = i + 1
        seq = per_kernel.get(kernel, [])
        if i >= len(seq):
            continue
        rec = ops.setdefault(op, {"bytes": 0.0, "ns": 0.0, "kernels": []})
        rec["bytes"] += seq[i][1]
        rec["ns"] += seq[i][2]
        rec["kernels"].append(kernel)
    pm = bs_perf()
    cw, tw = gen.WORKLOADS[capture], gen.WORKLOADS[target]
    out = {}
    for op in KERNEL_SRC:
        want = [k for k, o in STEP_KERNELS if o == op]
        if op not in ops or ops[op]["kernels"] != want:
            continue
        scale = (pm.moved_bytes(op, tw.NL, tw.NG, tw.NL) / pm.moved_bytes(op, cw.NL, cw.NG, cw.NL))
        out[op] = {"bytes_per_launch": ops[op]["bytes"] * scale, "config": target,
                   "measured_bytes": ops[op]["bytes"], "measured_us": ops[op]["ns"] / 1e3,
                   "measured_on": capture, "scale": scale, "kernels": want,
                   "src_sha256": src_sha(KERNEL_SRC[op])}
    doc = {"source": [os.path.basename(p) for p in paths],
           "note": f"dram__bytes_read.sum + dram__bytes_write.sum of each operation's kernels "
                   f"(first call in one bench step), measured on the {capture} mesh, one kernel "
                   f"family per ncu capture, scaled to the {target} mesh by the operation's "
                   "moved-bytes model", "kernels": out}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(doc, f, indent=1)
    print(json.dumps(doc, indent=1))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.traffic_from:
        return traffic_from_csv(args.traffic_from, args.traffic_capture, args.config)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.norm_ab:
        return run_norm_ab(args)
    if args.mass_operator:
        return run_mass_operator(args)
    if args.cg_solve:
        return run_cg_solve(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
