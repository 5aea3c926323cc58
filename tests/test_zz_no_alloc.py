"""The allocation-free inner product (bs_dot_noalloc) against the oracle.

bs_dot_noalloc serves callers that cannot call cudaMalloc -- code inside a
device-memory allocator's own hooks, or a runtime that owns all device
memory -- and so cannot create a context.  It keeps its reduction scratch in
a static device array shared by all calls.  Checked here through the C ABI:
its value against the oracle's Dot2 inner product within the reductions'
1e-12 relative bound, on two calls in a row; that calls after the first
allocate no device memory; and that the Python binding refuses operands on
another device.  This file is collected last so that a stop at the first
failure has already run every other test; it also passes on its own in a
fresh process.
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
import oracle  # noqa: E402
import order_fem_cg_gb300 as bs  # noqa: E402

DEV = torch.device("cuda", 0)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_c_abi(x, y, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return bs.lib.bs_dot_noalloc(x.numel(), _ptr(x), _ptr(y), _ptr(out), stream)


def _close(got, ref):
    return abs(got - ref) <= 1e-12 * abs(ref) or (ref == 0.0 and got == 0.0)


@pytest.mark.parametrize("n,off", [(3_000_017, 0), (1 << 20, 1), (5, 0), (0, 0)])
def test_noalloc_dot_matches_oracle_on_two_calls(n, off):
    torch.cuda.set_device(0)
    xh = gen.uniform_pm1(31, 7, n + off)[off:]
    yh = gen.uniform_pm1(31, 9, n + off)[off:]
    xb = torch.from_numpy(gen.uniform_pm1(31, 7, n + off)).to(DEV)
    yb = torch.from_numpy(gen.uniform_pm1(31, 9, n + off)).to(DEV)
    x, y = xb[off:], yb[off:]
    ref = oracle.dot(xh, yh)
    out = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    for _ in range(2):
        out.fill_(float("nan"))
        assert _call_c_abi(x, y, out) == bs.BS_OK
        torch.cuda.synchronize()
        assert _close(out.cpu().item(), ref)


def test_noalloc_dot_back_to_back_sizes():
    """The shared array keeps the last call's contents: a large call, then a
    small one, then a large one again, all queued before any sync."""
    torch.cuda.set_device(0)
    sizes = [2_500_001, 77, 2_500_001]
    xh = [gen.uniform_pm1(41, 3, n) for n in sizes]
    yh = [gen.uniform_pm1(41, 4, n) for n in sizes]
    xs = [torch.from_numpy(a).to(DEV) for a in xh]
    ys = [torch.from_numpy(a).to(DEV) for a in yh]
    outs = [torch.empty(1, dtype=torch.float64, device=DEV) for _ in sizes]
    for x, y, o in zip(xs, ys, outs):
        assert _call_c_abi(x, y, o) == bs.BS_OK
    torch.cuda.synchronize()
    for a, b, o in zip(xh, yh, outs):
        assert _close(o.cpu().item(), oracle.dot(a, b))


def test_noalloc_dot_allocates_nothing():
    """After a first call (which may load the library's device code), calls
    leave the device's free memory and torch's allocator untouched: a
    cudaMalloc of any size would take at least one 2 MB page."""
    torch.cuda.set_device(0)
    n = 4_000_000
    x = torch.from_numpy(gen.uniform_pm1(51, 1, n)).to(DEV)
    y = torch.from_numpy(gen.uniform_pm1(51, 2, n)).to(DEV)
    out = torch.empty(1, dtype=torch.float64, device=DEV)
    assert _call_c_abi(x, y, out) == bs.BS_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(DEV)
    alloc0 = torch.cuda.memory_allocated(DEV)
    for _ in range(5):
        assert _call_c_abi(x, y, out) == bs.BS_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(DEV)
    assert free1 == free0 and torch.cuda.memory_allocated(DEV) == alloc0
    assert _close(out.cpu().item(), oracle.dot(gen.uniform_pm1(51, 1, n), gen.uniform_pm1(51, 2, n)))


def test_noalloc_binding_rejects_host_tensors():
    x = torch.zeros(8, dtype=torch.float64)
    out = torch.empty(1, dtype=torch.float64, device=DEV)
    with pytest.raises(TypeError):
        bs.bs_dot_noalloc(x, x, out)


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two CUDA devices")
def test_noalloc_binding_rejects_other_device():
    torch.cuda.set_device(0)
    x = torch.zeros(8, dtype=torch.float64, device="cuda:1")
    out = torch.empty(1, dtype=torch.float64, device=DEV)
    with pytest.raises(ValueError):
        bs.bs_dot_noalloc(x, x, out)
