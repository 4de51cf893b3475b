"""osf_softmax_rows_noalloc, called through the C ABI, against the oracle and osf_softmax_rows.

The no-allocation entry point serves callers that cannot call cudaMalloc (for example code
running during CUDA graph capture, or a library given only its input and output buffers).  It
must give the same result as the workspace-taking entry point and as the fp64 oracle, on two
calls in a row (the shared scratch array keeps the previous call's contents), and refuse problems
larger than its fixed scratch.  This file is collected last so a failure here cannot hide
earlier tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import F32_ATOL, SUM_TOL, assert_f32_close, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def noalloc_fn(osf):
    fn = osf.lib().osf_softmax_rows_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_void_p]
    return fn


@pytest.mark.parametrize("rows,T", [(1, 1 << 22), (3, 100003), (7, 32768), (2, 40001)])
def test_noalloc_matches_oracle_and_workspace_entry_point(osf, rows, T):
    fn = noalloc_fn(osf)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):   # two calls in a row: the shared scratch holds the previous call's states
        xh = si.softmax_rows_input(rows, T, seed=100 * call + rows)
        x = f32_tensor(xh)
        ref = osf.osf_softmax_rows(x)
        z = torch.full_like(x, float("nan"))
        st = fn(x.data_ptr(), z.data_ptr(), rows, T, stream)
        assert st == osf.OSF_OK, osf.osf_status_string(st)
        torch.cuda.synchronize()
        got = z.cpu().numpy()
        assert_f32_close(got, oracle.softmax(xh), what=f"call {call} against the oracle")
        diff = float((z - ref).abs().max())
        assert diff <= F32_ATOL, f"call {call}: max abs difference {diff:.3e} to osf_softmax_rows"
        sums = got.astype(np.float64).sum(axis=-1)
        assert float(np.max(np.abs(sums - 1.0))) <= SUM_TOL
    assert osf.osf_device_status() == osf.OSF_OK


def test_noalloc_in_place(osf):
    fn = noalloc_fn(osf)
    xh = si.softmax_rows_input(1, 1 << 20, seed=5)
    x = f32_tensor(xh)
    st = fn(x.data_ptr(), x.data_ptr(), 1, 1 << 20, torch.cuda.current_stream().cuda_stream)
    assert st == osf.OSF_OK
    torch.cuda.synchronize()
    assert_f32_close(x.cpu().numpy(), oracle.softmax(xh), what="in place")


@pytest.mark.parametrize("rows,T", [(1, 1 << 22), (3, 100003)])
def test_noalloc_captured_in_a_graph(osf, rows, T):
    """The documented use: one eager call first (it looks up the array on this device), then the
    entry point inside a captured CUDA graph, whose replay must equal the eager result bit for bit
    (the kernels are deterministic)."""
    fn = noalloc_fn(osf)
    x = f32_tensor(si.softmax_rows_input(rows, T, seed=77))
    z = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert fn(x.data_ptr(), z.data_ptr(), rows, T, side.cuda_stream) == osf.OSF_OK
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = z.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = fn(x.data_ptr(), z.data_ptr(), rows, T, torch.cuda.current_stream().cuda_stream)
    assert st == osf.OSF_OK
    z.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, z)


def test_noalloc_rejects_oversize_and_bad_arguments(osf):
    fn = noalloc_fn(osf)
    s = torch.cuda.current_stream().cuda_stream
    big_rows, big_T = 20000, 40000            # one chunk state per row: 20000 > 16384
    x = ctypes.c_void_p(1 << 40)
    z = ctypes.c_void_p(1 << 44)
    before = osf.osf_launch_count()
    assert fn(x, z, big_rows, big_T, s) == osf.OSF_ERR_WORKSPACE
    assert fn(x, z, -1, 4, s) == osf.OSF_ERR_INVALID
    assert fn(None, z, 2, 4, s) == osf.OSF_ERR_INVALID
    assert fn(x, ctypes.c_void_p((1 << 40) + 8), 2, 4, s) == osf.OSF_ERR_INVALID
    assert fn(None, None, 0, 4, s) == osf.OSF_OK
    assert osf.osf_launch_count() == before   # nothing launched
