"""The allocation-free inner product (bs_dot_noalloc) against bs_dot.

bs_dot_noalloc serves callers that cannot call cudaMalloc (allocator hooks,
host callbacks, runtimes that own all device memory) and so cannot create a
context.  It keeps its reduction scratch in a static device array shared by
all calls.  This file is collected last so that a stop at the first failure
has already run every other test; it also passes on its own in a fresh
process.  Tolerance: the reductions' 1e-12 relative bound.
"""

import ctypes

import numpy as np
import pytest

import bsinputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from conftest import build_lib  # noqa: E402

build_lib()
import order_fem_cg_gb300 as bs  # noqa: E402

DEV = torch.device("cuda", 0)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_c_abi(x, y, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return bs.lib.bs_dot_noalloc(x.numel(), _ptr(x), _ptr(y), _ptr(out), stream)


@pytest.mark.parametrize("n,off", [(3_000_017, 0), (1 << 20, 1), (5, 0), (0, 0)])
def test_noalloc_dot_matches_dot_on_two_calls(n, off):
    torch.cuda.set_device(0)
    xb = torch.from_numpy(gen.uniform_pm1(31, 7, n + off)).to(DEV)
    yb = torch.from_numpy(gen.uniform_pm1(31, 9, n + off)).to(DEV)
    x, y = xb[off:], yb[off:]
    ref = bs.bs_dot(x, y).cpu().item()
    out = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    for _ in range(2):
        out.fill_(float("nan"))
        assert _call_c_abi(x, y, out) == bs.BS_OK
        torch.cuda.synchronize()
        got = out.cpu().item()
        assert abs(got - ref) <= 1e-12 * abs(ref) or (ref == 0.0 and got == 0.0)


def test_noalloc_dot_back_to_back_sizes():
    """The shared array keeps the last call's contents: a large call, then a
    small one, then a large one again, all queued before any sync."""
    torch.cuda.set_device(0)
    sizes = [2_500_001, 77, 2_500_001]
    xs = [torch.from_numpy(gen.uniform_pm1(41, 3, n)).to(DEV) for n in sizes]
    ys = [torch.from_numpy(gen.uniform_pm1(41, 4, n)).to(DEV) for n in sizes]
    outs = [torch.empty(1, dtype=torch.float64, device=DEV) for _ in sizes]
    for x, y, o in zip(xs, ys, outs):
        assert _call_c_abi(x, y, o) == bs.BS_OK
    torch.cuda.synchronize()
    for x, y, o in zip(xs, ys, outs):
        ref = bs.bs_dot(x, y).cpu().item()
        assert abs(o.cpu().item() - ref) <= 1e-12 * abs(ref)
