"""GB300 Benchmark Streaming library: Python binding of libbs.so.

Thin ctypes marshalling over the C ABI declared in ``include/bs.h``; every
operation runs in the library's sm_103a kernels.  Torch tensors supply
device memory and the CUDA stream (the current stream unless one is given).
The binding has the C ABI's names:

    bs_copy, bs_axpy, bs_norm, bs_dot, bs_cg_update      (BS1-BS5)
    bs_gather, bs_scatter, bs_cg_iteration                (BS6, BS7, one CG pass)
    Mesh (bs_mesh_build_box & co), DeviceTables (bs_gs_dev)

If libbs.so is missing or fails to load, importing the binding raises: there
is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbs.so")

BS_OK = 0
BS_EINVAL = -1
BS_ECUDA = -2
BS_ENOMEM = -3
BS_EBOUNDS = -4
BS_EALIGN = -5
BS_ETIMEOUT = -6

SHUFFLE_ELEMS = 1
PERMUTE_GLOBAL = 2
MASK_BOUNDARY = 4
ROTATE_ELEMS = 8
GATHER_SEG_MAX = 4096
GATHER_SEG_DEFAULT = 2048
ONEPASS_SCATTER_BYTES = 32 << 20   # include/bs.h: BS_ONEPASS_SCATTER_BYTES
ONEPASS_GATHER_BYTES = 8 << 20     # include/bs.h: BS_ONEPASS_GATHER_BYTES


def gs_launches(NL, NG, planned):
    """(gather, scatter) kernel launches of one bs_gather / bs_scatter call
    with a context created under the current environment."""
    if not planned:
        return 1, 1
    small = os.environ.get("BS_TUNE_ONEPASS", "1") != "0"
    return (1 if small and 8 * NL <= ONEPASS_GATHER_BYTES else 2,
            1 if small and 8 * NG <= ONEPASS_SCATTER_BYTES else 2)

# Every symbol include/bs.h declares.
EXPORTS = (
    "bs_strerror", "bs_last_error", "bs_ctx_create", "bs_ctx_destroy", "bs_ctx_num_sms",
    "bs_ctx_device_status", "bs_copy", "bs_axpy", "bs_norm", "bs_dot", "bs_cg_update",
    "bs_mesh_build_box", "bs_mesh_build_box_ex", "bs_mesh_info", "bs_mesh_tables",
    "bs_mesh_validate", "bs_mesh_destroy", "bs_gather", "bs_scatter", "bs_cg_iteration",
    "bs_dot_noalloc", "bs_mesh_plan", "bs_mesh_plan_info", "bs_mesh_plan_tables",
    "bs_apply_diag", "bs_axpy_dev", "bs_cg_solve", "bs_cg_solve_fused", "bs_probe_grid_barrier",
    "bs_mesh_from_ids",
)


class BSError(RuntimeError):
    def __init__(self, status, msg=""):
        self.status = status
        super().__init__(f"{_strerror(status)} ({status}): {msg}")


class MeshInfo(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("N", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("max_row", ctypes.c_int32), ("K", ctypes.c_int64), ("NL", ctypes.c_int64),
                ("NG", ctypes.c_int64), ("nnz", ctypes.c_int64), ("nblocks", ctypes.c_int64),
                ("seg_max", ctypes.c_int32), ("seg_target", ctypes.c_int32)]


_PLAN_INTS = ("cluster", "s_ntiles", "s_nbuckets", "s_tile_rows", "s_bucket_len", "g_ntiles",
              "g_nbuckets", "g_tile_len", "g_bucket_entries_max", "g_bucket_rows_max", "g_mmax")
PLAN_TABLES = ("s_tileRows", "s_runStart", "s_src", "s_dst", "g_subRows", "g_tileSlot",
               "g_runStart", "g_src", "g_pos", "g_groupStart", "g_rowPos")


class PlanDev(ctypes.Structure):
    _fields_ = ([(k, ctypes.c_int32) for k in _PLAN_INTS]
                + [(k, ctypes.c_void_p) for k in PLAN_TABLES]
                + [("work", ctypes.c_void_p), ("work_len", ctypes.c_int64)])


class PlanInfo(ctypes.Structure):
    _fields_ = ([(k, ctypes.c_int32) for k in (
        "valid", "cluster", "s_tile_rows", "s_bucket_len", "g_tile_len", "g_bucket_entries",
        "s_ntiles", "s_nbuckets", "g_ntiles", "g_nbuckets", "g_bucket_rows_max",
        "g_bucket_entries_max", "g_mmax", "reserved")]
        + [(k, ctypes.c_int64) for k in ("smem_s1", "smem_s2", "smem_g1", "smem_g2")])


class GSDev(ctypes.Structure):
    _fields_ = [("NL", ctypes.c_int64), ("NG", ctypes.c_int64), ("nnz", ctypes.c_int64),
                ("nblocks", ctypes.c_int64), ("seg_max", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("scatterIds", ctypes.c_void_p),
                ("rowStarts", ctypes.c_void_p), ("localIds", ctypes.c_void_p),
                ("blockStarts", ctypes.c_void_p), ("plan", ctypes.c_void_p)]


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double


def _declare(lib):
    sig = {
        "bs_strerror": ([_int], ctypes.c_char_p),
        "bs_last_error": ([_vp], ctypes.c_char_p),
        "bs_ctx_create": ([_int, ctypes.POINTER(_vp)], _int),
        "bs_ctx_destroy": ([_vp], _int),
        "bs_ctx_num_sms": ([_vp], _int),
        "bs_ctx_device_status": ([_vp, _vp, ctypes.POINTER(_int)], _int),
        "bs_copy": ([_vp, _i64, _vp, _vp, _vp], _int),
        "bs_axpy": ([_vp, _i64, _dbl, _vp, _dbl, _vp, _vp], _int),
        "bs_norm": ([_vp, _i64, _vp, _vp, _vp], _int),
        "bs_dot": ([_vp, _i64, _vp, _vp, _vp, _vp], _int),
        "bs_cg_update": ([_vp, _i64, _vp, _vp, _dbl, _vp, _vp, _vp, _vp, _vp, _vp], _int),
        "bs_mesh_build_box": ([_int, _int, ctypes.c_uint64, ctypes.c_uint32,
                               ctypes.POINTER(_vp)], _int),
        "bs_mesh_build_box_ex": ([_int, _int, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                  ctypes.POINTER(_vp)], _int),
        "bs_mesh_info": ([_vp, ctypes.POINTER(MeshInfo)], _int),
        "bs_mesh_tables": ([_vp] + [ctypes.POINTER(_vp)] * 4, _int),
        "bs_mesh_validate": ([_vp], _int),
        "bs_mesh_destroy": ([_vp], _int),
        "bs_gather": ([_vp, ctypes.POINTER(GSDev), _vp, _vp, _vp], _int),
        "bs_scatter": ([_vp, ctypes.POINTER(GSDev), _vp, _vp, _vp], _int),
        "bs_cg_iteration": ([_vp, ctypes.POINTER(GSDev)] + [_vp] * 10, _int),
        "bs_apply_diag": ([_vp, ctypes.POINTER(GSDev), _vp, _vp, _vp, _vp], _int),
        "bs_axpy_dev": ([_vp, _i64, _dbl, _vp, _vp, _vp, _vp, _vp], _int),
        "bs_cg_solve": ([_vp, ctypes.POINTER(GSDev)] + [_vp] * 6 + [ctypes.c_int32, _vp, _vp],
                        _int),
        "bs_cg_solve_fused": ([_vp, ctypes.POINTER(GSDev)] + [_vp] * 7 +
                              [ctypes.c_int32, _vp, _vp], _int),
        "bs_probe_grid_barrier": ([_vp, _int, _vp], _int),
        "bs_mesh_from_ids": ([_i64, _i64, _vp, ctypes.c_int32, ctypes.POINTER(_vp)], _int),
        "bs_dot_noalloc": ([_i64, _vp, _vp, _vp, _vp], _int),
        "bs_mesh_plan": ([_vp] + [ctypes.c_int32] * 5, _int),
        "bs_mesh_plan_info": ([_vp, ctypes.POINTER(PlanInfo)], _int),
        "bs_mesh_plan_tables": ([_vp] + [ctypes.POINTER(_vp)] * 11, _int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built: run `python order_fem_cg_gb300/build.py` "
            "(nvcc for sm_103a); there is no non-CUDA implementation")
    lib = ctypes.CDLL(LIB_PATH)
    _declare(lib)
    return lib


lib = _load()


def _strerror(status):
    return lib.bs_strerror(int(status)).decode()


# ----------------------------------------------------------------- context

class Context:
    """A bs_ctx: one device, one stream at a time (owns the reduction workspace)."""

    def __init__(self, device=None):
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        h = _vp()
        st = lib.bs_ctx_create(self.device, ctypes.byref(h))
        if st != BS_OK:
            raise BSError(st, f"bs_ctx_create(device={self.device})")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib.bs_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_sms(self):
        return lib.bs_ctx_num_sms(self.handle)

    def check(self, st, what):
        if st != BS_OK:
            raise BSError(st, f"{what}: {lib.bs_last_error(self.handle).decode()}")

    def device_status(self, stream=None):
        out = _int(0)
        self.check(lib.bs_ctx_device_status(self.handle, _stream(stream), ctypes.byref(out)),
                   "bs_ctx_device_status")
        return out.value


_default_ctx = {}


def default_context(device=None):
    if device is None:
        device = torch.cuda.current_device()
    ctx = _default_ctx.get(device)
    if ctx is None:
        ctx = _default_ctx[device] = Context(device)
    return ctx


def _stream(stream):
    if stream is None:
        return _vp(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return _vp(stream.cuda_stream)
    return _vp(int(stream))


def _vec(t, name, n=None):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float64 or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA float64 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if n is not None and t.numel() != n:
        raise ValueError(f"{name}: expected {n} elements, got {t.numel()}")
    return _vp(t.data_ptr())


def _scalar_out(out, device):
    if out is None:
        out = torch.empty(1, dtype=torch.float64, device=device)
    _vec(out, "out")
    return out


def _ctx(ctx, t):
    return ctx if ctx is not None else default_context(t.device.index)


# ------------------------------------------------------------ BS1 - BS5

def bs_copy(x, y, stream=None, ctx=None):
    """BS1: y <- x."""
    ctx = _ctx(ctx, x)
    ctx.check(lib.bs_copy(ctx.handle, x.numel(), _vec(x, "x"), _vec(y, "y", x.numel()),
                          _stream(stream)), "bs_copy")
    return y


def bs_axpy(alpha, x, beta, y, stream=None, ctx=None):
    """BS2: y <- fma(alpha, x, beta * y)."""
    ctx = _ctx(ctx, x)
    ctx.check(lib.bs_axpy(ctx.handle, x.numel(), float(alpha), _vec(x, "x"), float(beta),
                          _vec(y, "y", x.numel()), _stream(stream)), "bs_axpy")
    return y


def bs_axpy_dev(alpha, x, beta_num, beta_den, y, stream=None, ctx=None):
    """BS2 with beta = beta_num[0] / beta_den[0] formed on the device (0 if
    the denominator is 0): y <- fma(alpha, x, beta * y)."""
    ctx = _ctx(ctx, x)
    ctx.check(lib.bs_axpy_dev(ctx.handle, x.numel(), float(alpha), _vec(x, "x"),
                              _vec(beta_num, "beta_num"), _vec(beta_den, "beta_den"),
                              _vec(y, "y", x.numel()), _stream(stream)), "bs_axpy_dev")
    return y


def bs_norm(x, out=None, stream=None, ctx=None):
    """BS3: out[0] <- x . x (squared 2-norm), on the device."""
    ctx = _ctx(ctx, x)
    out = _scalar_out(out, x.device)
    ctx.check(lib.bs_norm(ctx.handle, x.numel(), _vec(x, "x"), _vp(out.data_ptr()),
                          _stream(stream)), "bs_norm")
    return out


def bs_dot(x, y, out=None, stream=None, ctx=None):
    """BS4: out[0] <- x . y, on the device."""
    ctx = _ctx(ctx, x)
    out = _scalar_out(out, x.device)
    ctx.check(lib.bs_dot(ctx.handle, x.numel(), _vec(x, "x"), _vec(y, "y", x.numel()),
                         _vp(out.data_ptr()), _stream(stream)), "bs_dot")
    return out


def bs_cg_update(p, Ap, x, r, alpha=0.0, alpha_num=None, alpha_den=None, rdotr=None,
                 reduce=True, stream=None, ctx=None):
    """BS5: x += alpha p; r -= alpha Ap; rdotr[0] <- r . r (updated r).

    alpha is the float `alpha`, or alpha_num[0] / alpha_den[0] (device
    scalars) when both are given.  Returns rdotr (None if reduce=False).
    """
    ctx = _ctx(ctx, p)
    n = p.numel()
    if reduce:
        rdotr = _scalar_out(rdotr, p.device)
    num = _vec(alpha_num, "alpha_num") if alpha_num is not None else _vp(0)
    den = _vec(alpha_den, "alpha_den") if alpha_den is not None else _vp(0)
    ctx.check(lib.bs_cg_update(ctx.handle, n, num, den, float(alpha), _vec(p, "p"),
                               _vec(Ap, "Ap", n), _vec(x, "x", n), _vec(r, "r", n),
                               _vp(rdotr.data_ptr()) if reduce else _vp(0), _stream(stream)),
              "bs_cg_update")
    return rdotr if reduce else None


def bs_dot_noalloc(x, y, out, stream=None):
    """BS4 without a context: for callers that cannot allocate device memory.

    Same result as bs_dot, with the reduction's scratch in a static device
    array shared by all calls (serialise calls; `out` must be preallocated).
    x, y and out must live on the current CUDA device: the call launches
    there and has no context to check against.
    """
    cur = torch.cuda.current_device()
    for name, t in (("x", x), ("y", y), ("out", out)):
        if isinstance(t, torch.Tensor) and t.is_cuda and t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{cur}")
    st = lib.bs_dot_noalloc(x.numel(), _vec(x, "x"), _vec(y, "y", x.numel()), _vec(out, "out", 1),
                            _stream(stream))
    if st != BS_OK:
        raise BSError(st, "bs_dot_noalloc")
    return out


# ------------------------------------------------------------- mesh

class Mesh:
    """Mesh index tables built on the host (bs_mesh_*): a box hex mesh, or
    any mesh given by its local-to-global table (Mesh.from_ids)."""

    def __init__(self, E, N, seed, flags=SHUFFLE_ELEMS | PERMUTE_GLOBAL, seg_target=None):
        h = _vp()
        if seg_target is None:
            st = lib.bs_mesh_build_box(int(E), int(N), int(seed), int(flags), ctypes.byref(h))
        else:
            st = lib.bs_mesh_build_box_ex(int(E), int(N), int(seed), int(flags), int(seg_target),
                                          ctypes.byref(h))
        if st != BS_OK:
            raise BSError(st, f"bs_mesh_build_box(E={E}, N={N})")
        self._adopt(h)

    def _adopt(self, h):
        self.handle = h
        info = MeshInfo()
        lib.bs_mesh_info(h, ctypes.byref(info))
        self.info = info

    @classmethod
    def from_ids(cls, scatter_ids, NG, seg_target=None):
        """Tables of any mesh from its local-to-global table (int32, -1 =
        masked, entries < NG)."""
        ids = np.ascontiguousarray(scatter_ids, dtype=np.int32)
        h = _vp()
        st = lib.bs_mesh_from_ids(ids.size, int(NG), ids.ctypes.data,
                                  int(seg_target or GATHER_SEG_DEFAULT), ctypes.byref(h))
        if st != BS_OK:
            raise BSError(st, f"bs_mesh_from_ids(NL={ids.size}, NG={NG})")
        self = cls.__new__(cls)
        self._adopt(h)
        return self

    def __del__(self):
        if getattr(self, "handle", None):
            lib.bs_mesh_destroy(self.handle)
            self.handle = None

    def __getattr__(self, k):
        if k in ("E", "N", "flags", "max_row", "K", "NL", "NG", "nnz", "nblocks", "seg_max",
                 "seg_target"):
            return getattr(self.info, k)
        raise AttributeError(k)

    def validate(self):
        return lib.bs_mesh_validate(self.handle)

    def tables(self):
        """Copies of the four host tables as int32 numpy arrays."""
        ptrs = [_vp() for _ in range(4)]
        st = lib.bs_mesh_tables(self.handle, *[ctypes.byref(p) for p in ptrs])
        if st != BS_OK:
            raise BSError(st, "bs_mesh_tables")
        sizes = (self.NL, self.NG + 1, self.nnz, self.nblocks + 1)
        out = {}
        for name, p, n in zip(("scatterIds", "rowStarts", "localIds", "blockStarts"), ptrs, sizes):
            if n == 0:
                out[name] = np.zeros(0, dtype=np.int32)
            else:
                buf = (ctypes.c_int32 * n).from_address(p.value)
                out[name] = np.frombuffer(buf, dtype=np.int32).copy()
        return out

    def plan(self, s_tile_rows, s_bucket_len, g_tile_len, g_bucket_entries, cluster=2):
        """Rebuild the two-pass plan with other per-block sizes / cluster size (returns the status)."""
        return lib.bs_mesh_plan(self.handle, int(s_tile_rows), int(s_bucket_len), int(g_tile_len),
                                int(g_bucket_entries), int(cluster))

    def plan_info(self):
        info = PlanInfo()
        lib.bs_mesh_plan_info(self.handle, ctypes.byref(info))
        return info

    def plan_tables(self):
        """Copies of the plan's host tables (int32 / uint16 numpy arrays), or None."""
        pi = self.plan_info()
        if not pi.valid:
            return None
        ptrs = [_vp() for _ in PLAN_TABLES]
        st = lib.bs_mesh_plan_tables(self.handle, *[ctypes.byref(p) for p in ptrs])
        if st != BS_OK:
            raise BSError(st, "bs_mesh_plan_tables")
        sizes = {"s_tileRows": (pi.s_ntiles + 1, np.int32),
                 "s_runStart": ((pi.s_ntiles + 1) * pi.s_nbuckets, np.int32),
                 "s_src": (self.nnz, np.uint16), "s_dst": (self.nnz, np.uint16),
                 "g_subRows": (pi.cluster * pi.g_nbuckets + 1, np.int32),
                 "g_tileSlot": (pi.g_ntiles + 1, np.int32),
                 "g_runStart": ((pi.g_ntiles + 1) * pi.g_nbuckets, np.int32),
                 "g_src": (self.nnz, np.uint16), "g_pos": (self.nnz, np.uint16),
                 "g_groupStart": (pi.cluster * pi.g_nbuckets * (pi.g_mmax + 1), np.uint16),
                 "g_rowPos": (self.NG, np.uint16)}
        out = {}
        for name, p in zip(PLAN_TABLES, ptrs):
            n, dt = sizes[name]
            if n == 0:
                out[name] = np.zeros(0, dtype=dt)
            else:
                ct = ctypes.c_int32 if dt == np.int32 else ctypes.c_uint16
                out[name] = np.frombuffer((ct * n).from_address(p.value), dtype=dt).copy()
        return out

    def to_device(self, device=None, planned=True):
        """Upload the tables; with planned=True (and a valid plan) also the
        two-pass plan and its work buffer, so bs_gather/bs_scatter use it."""
        plan = None
        if planned:
            pt = self.plan_tables()
            if pt is not None:
                plan = (pt, self.plan_info())
        return DeviceTables.from_host(self.tables(), self.info, device, plan)


class DeviceTables:
    """Index tables resident in device memory plus the bs_gs_dev struct."""

    def __init__(self, scatterIds, rowStarts, localIds, blockStarts, NL, NG, nnz, nblocks,
                 seg_max):
        self.scatterIds, self.rowStarts = scatterIds, rowStarts
        self.localIds, self.blockStarts = localIds, blockStarts
        self.NL, self.NG, self.nnz, self.nblocks, self.seg_max = NL, NG, nnz, nblocks, seg_max
        for name in ("scatterIds", "rowStarts", "localIds", "blockStarts"):
            t = getattr(self, name)
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise TypeError(f"{name}: expected a contiguous CUDA int32 tensor")

        def ptr(t):
            return t.data_ptr() if t.numel() else 0

        self.struct = GSDev(NL, NG, nnz, nblocks, seg_max, 0, ptr(scatterIds), ptr(rowStarts),
                            ptr(localIds), ptr(blockStarts), None)
        self.plan = None
        self.plan_struct = None

    def attach_plan(self, tabs, pinfo):
        """Upload a two-pass plan (host tables + PlanInfo) and allocate its work buffer."""
        dev = self.scatterIds.device
        up = {}
        for k in PLAN_TABLES:
            a = np.ascontiguousarray(tabs[k])
            if a.dtype == np.uint16:
                a = a.view(np.int16)        # same bits; torch has no general uint16 kernels
            up[k] = torch.from_numpy(a).to(dev)
        # 2 nnz: bs_apply_diag needs a second work array
        work = torch.empty(max(2 * self.nnz, 1), dtype=torch.float64, device=dev)
        ints = dict(cluster=pinfo.cluster, s_ntiles=pinfo.s_ntiles, s_nbuckets=pinfo.s_nbuckets,
                    s_tile_rows=pinfo.s_tile_rows, s_bucket_len=pinfo.s_bucket_len,
                    g_ntiles=pinfo.g_ntiles, g_nbuckets=pinfo.g_nbuckets,
                    g_tile_len=pinfo.g_tile_len, g_bucket_entries_max=pinfo.g_bucket_entries_max,
                    g_bucket_rows_max=pinfo.g_bucket_rows_max, g_mmax=pinfo.g_mmax)
        ps = PlanDev(**ints, **{k: (up[k].data_ptr() if up[k].numel() else 0) for k in PLAN_TABLES},
                     work=work.data_ptr(), work_len=2 * self.nnz)
        self.plan = dict(up, work=work, info=pinfo)
        self.plan_struct = ps
        self.struct.plan = ctypes.addressof(ps)
        return self

    def detach_plan(self):
        self.struct.plan = None
        self.plan = None
        self.plan_struct = None
        return self

    @classmethod
    def from_host(cls, tabs, info, device=None, plan=None):
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        up = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).to(dev)
              for k, v in tabs.items()}
        t = cls(up["scatterIds"], up["rowStarts"], up["localIds"], up["blockStarts"],
                int(info.NL), int(info.NG), int(info.nnz), int(info.nblocks), int(info.seg_max))
        if plan is not None:
            t.attach_plan(*plan)
        return t

    @property
    def device(self):
        return self.scatterIds.device

    @property
    def nbytes(self):
        n = sum(t.numel() * 4 for t in (self.scatterIds, self.rowStarts, self.localIds,
                                         self.blockStarts))
        if self.plan is not None:
            n += sum(self.plan[k].numel() * self.plan[k].element_size() for k in PLAN_TABLES)
        return n


# ------------------------------------------------------------ BS6 / BS7

def bs_gather(tables, qL, qG, stream=None, ctx=None):
    """BS6: qG <- Z^T qL (each global node's local copies summed in ascending local index)."""
    ctx = _ctx(ctx, qL)
    ctx.check(lib.bs_gather(ctx.handle, ctypes.byref(tables.struct), _vec(qL, "qL", tables.NL),
                            _vec(qG, "qG", tables.NG), _stream(stream)), "bs_gather")
    return qG


def bs_scatter(tables, qG, qL, stream=None, ctx=None):
    """BS7: qL <- Z qG (masked locals get +0.0)."""
    ctx = _ctx(ctx, qG)
    ctx.check(lib.bs_scatter(ctx.handle, ctypes.byref(tables.struct), _vec(qG, "qG", tables.NG),
                             _vec(qL, "qL", tables.NL), _stream(stream)), "bs_scatter")
    return qL


def bs_apply_diag(tables, xG, dL, yG, stream=None, ctx=None):
    """yG <- Z^T (dL .* (Z xG)): the global operator of a diagonal local operator
    (fused); dL None is the identity local operator (yG <- Z^T Z xG)."""
    ctx = _ctx(ctx, xG)
    ctx.check(lib.bs_apply_diag(ctx.handle, ctypes.byref(tables.struct), _vec(xG, "xG", tables.NG),
                                _vec(dL, "dL", tables.NL) if dL is not None else _vp(0),
                                _vec(yG, "yG", tables.NG), _stream(stream)), "bs_apply_diag")
    return yG


def bs_cg_solve(tables, dL, bG, xG, rG, pG, ApG, iters, scal=None, stream=None, ctx=None):
    """`iters` CG iterations on A = Z^T diag(dL) Z (dL None: Z^T Z), from xG
    (updated in place), every scalar on the device.  Returns scal
    [2 iters + 1]: rr_0 .. rr_iters, then pAp_0 .. pAp_{iters-1}."""
    ctx = _ctx(ctx, bG)
    NG = tables.NG
    iters = int(iters)
    if scal is None:
        scal = torch.empty(2 * iters + 1, dtype=torch.float64, device=bG.device)
    ctx.check(lib.bs_cg_solve(
        ctx.handle, ctypes.byref(tables.struct),
        _vec(dL, "dL", tables.NL) if dL is not None else _vp(0), _vec(bG, "bG", NG),
        _vec(xG, "xG", NG), _vec(rG, "rG", NG), _vec(pG, "pG", NG), _vec(ApG, "ApG", NG),
        iters, _vec(scal, "scal", 2 * iters + 1), _stream(stream)), "bs_cg_solve")
    return scal


def bs_probe_grid_barrier(absent_block=-1, stream=None, ctx=None):
    """Run the fused solve's grid barrier twice; with absent_block >= 0 that
    block never arrives and the others' bounded waits run out.  Returns the
    device status (BS_OK or BS_ETIMEOUT)."""
    ctx = ctx if ctx is not None else default_context()
    ctx.check(lib.bs_probe_grid_barrier(ctx.handle, int(absent_block), _stream(stream)),
              "bs_probe_grid_barrier")
    return ctx.device_status(stream)


def bs_cg_solve_fused(tables, dL, bG, xG, rG, pG, ApG, pL, iters, scal=None, stream=None,
                      ctx=None):
    """bs_cg_solve's iteration in one cooperative kernel (grid barriers, no
    launch per iteration) for launch-bound mesh sizes; pL [NL] is scratch."""
    ctx = _ctx(ctx, bG)
    NG = tables.NG
    iters = int(iters)
    if scal is None:
        scal = torch.empty(2 * iters + 1, dtype=torch.float64, device=bG.device)
    ctx.check(lib.bs_cg_solve_fused(
        ctx.handle, ctypes.byref(tables.struct),
        _vec(dL, "dL", tables.NL) if dL is not None else _vp(0), _vec(bG, "bG", NG),
        _vec(xG, "xG", NG), _vec(rG, "rG", NG), _vec(pG, "pG", NG), _vec(ApG, "ApG", NG),
        _vec(pL, "pL", tables.NL), iters, _vec(scal, "scal", 2 * iters + 1), _stream(stream)),
        "bs_cg_solve_fused")
    return scal


def bs_cg_iteration(tables, pG, pL, ApG, xG, rG, rr, pAp, rr_new, rnorm, stream=None, ctx=None):
    """One CG iteration's streaming sequence (identity local operator):
    scatter, gather, dot, fused update with alpha = rr/pAp on the device, norm."""
    ctx = _ctx(ctx, pG)
    NG, NL = tables.NG, tables.NL
    ctx.check(lib.bs_cg_iteration(
        ctx.handle, ctypes.byref(tables.struct), _vec(pG, "pG", NG), _vec(pL, "pL", NL),
        _vec(ApG, "ApG", NG), _vec(xG, "xG", NG), _vec(rG, "rG", NG), _vec(rr, "rr", 1),
        _vec(pAp, "pAp", 1), _vec(rr_new, "rr_new", 1), _vec(rnorm, "rnorm", 1),
        _stream(stream)), "bs_cg_iteration")
