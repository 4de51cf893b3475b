"""GPU parity of the streaming row softmax against the fp64 oracle, through the C ABI binding.

Workloads: rows of 8 * N(0, 1) with a +30 spike at a seeded column; the full-size
[4096, 32768] matrix and the 1-D vector of 2^26 elements are checked element by element.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import SUM_TOL, assert_f32_close, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def run(osf, x, inplace=False):
    xt = f32_tensor(x)
    z = osf.osf_softmax_rows(xt, xt if inplace else None)
    return z.cpu().numpy()


def check_rows(z, ref, what):
    assert_f32_close(z, ref, what=what)
    sums = z.astype(np.float64).sum(axis=-1)
    err = float(np.max(np.abs(sums - 1.0)))
    assert err <= SUM_TOL, f"{what}: row sum off by {err:.2e}"


def test_softmax_rows_full_size(osf):
    x = si.softmax_rows_input(4096, 32768, seed=0)
    z = run(osf, x)
    check_rows(z, oracle.softmax(x), "rows 4096x32768")


def test_softmax_1d_full_size(osf):
    x = si.softmax_rows_input(1, 1 << 26, seed=0)
    z = run(osf, x)
    ref = oracle.softmax(x)
    check_rows(z, ref, "1-D 2^26")
    big = ref > 1e-30
    rel = float(np.max(np.abs(z[big] - ref[big]) / ref[big]))
    assert rel <= 1e-5, f"1-D relative error {rel:.2e}"


@pytest.mark.parametrize("rows", [1, 3, 64])
@pytest.mark.parametrize("T", [1, 3, 4, 100, 1000, 4096, 8196, 20004, 32767, 32768, 32772, 100003])
def test_softmax_shapes(osf, rows, T):
    x = si.softmax_rows_input(rows, T, seed=rows * 7 + T)
    check_rows(run(osf, x), oracle.softmax(x), f"rows={rows} T={T}")


@pytest.mark.parametrize("T", [4096, 32768, 200000])
def test_softmax_in_place(osf, T):
    x = si.softmax_rows_input(5, T, seed=T)
    check_rows(run(osf, x, inplace=True), oracle.softmax(x), f"in place T={T}")


@pytest.mark.parametrize("T", [4096, 16384])
def test_softmax_special_rows(osf, T):
    x = np.zeros((5, T), dtype=np.float32)
    x[0] = 3.25                      # constant row -> uniform
    x[1] = -200.0                    # all very negative -> uniform (initial max must be -inf)
    x[2, 123] = 30.0                 # spike
    x[3] = -np.inf                   # masked logits ...
    x[3, :7] = np.arange(7)          # ... except seven
    x[4] = si.normal_f32((T,), 4, si.STREAM_X, 1e3)   # huge spread
    z = run(osf, x)
    check_rows(z, oracle.softmax(x), f"special rows T={T}")
    assert np.all(z[3, 7:] == 0)


def test_softmax_misaligned(osf):
    T = 1000
    x = si.softmax_rows_input(3, T, seed=1)
    buf = torch.empty(3 * T + 1, device="cuda")
    buf[1:] = f32_tensor(x).reshape(-1)
    xt = buf[1:].view(3, T)
    z = osf.osf_softmax_rows(xt).cpu().numpy()
    check_rows(z, oracle.softmax(x), "misaligned")


def test_softmax_guard_bands(osf):
    T, rows, g = 32768, 3, 1024
    x = si.softmax_rows_input(rows, T, seed=2)
    buf = torch.full((rows * T + 2 * g,), -5.0, device="cuda")
    z = buf[g:g + rows * T].view(rows, T)
    osf.osf_softmax_rows(f32_tensor(x), z)
    torch.cuda.synchronize()
    assert torch.all(buf[:g] == -5.0) and torch.all(buf[g + rows * T:] == -5.0)
    check_rows(z.cpu().numpy(), oracle.softmax(x), "guard bands")


def test_softmax_deterministic(osf):
    x = f32_tensor(si.softmax_rows_input(1, 1 << 22, seed=3))
    a = osf.osf_softmax_rows(x)
    b = osf.osf_softmax_rows(x)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
