"""GPU parity of ``osf_softmax_rows_ex`` (scaled, optionally causal row softmax on float32 /
bfloat16 strided rows) against ``oracle.softmax_masked`` on the same values.

Tolerances: float32 output as for ``osf_softmax_rows`` (max abs 1e-4, row sums 1e-5).  A
bfloat16 output is the float32 result rounded to nearest bfloat16, which is within 2^-9
relative; the test allows 4e-3 relative (twice that) and no absolute slack beyond 1e-30.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_f32_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def to_dev(x32, dtype, pad=0):
    t = torch.from_numpy(x32).cuda()
    rows, T = t.shape
    store = torch.zeros((rows, T + pad), dtype=dtype, device="cuda")
    store[:, :T] = t.to(dtype)
    return store[:, :T]


def values(t):
    return t.float().cpu().numpy().astype(np.float64)


def check(z, ref, what):
    got = values(z)
    if z.dtype == torch.bfloat16:
        err = np.abs(got - ref)
        bad = err > 4e-3 * np.abs(ref) + 1e-30
        assert not bad.any(), f"{what}: {bad.sum()} elements off, worst {err.max():.3g}"
    else:
        assert_f32_close(got, ref, atol=1e-4, what=what)
        assert np.abs(got.sum(axis=1) - (ref.sum(axis=1))).max() <= 1e-5, what + " row sums"


@pytest.mark.parametrize("T", [1, 7, 8, 100, 1000, 4096, 32768, 40000])
@pytest.mark.parametrize("dtypes", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
def test_dtypes_and_lengths(osf, T, dtypes):
    tin, tout = (torch.bfloat16 if d == "bf16" else torch.float32 for d in dtypes)
    rows = 3 if T > 30000 else 33
    x32 = si.softmax_rows_input(rows, T, seed=T)
    x = to_dev(x32, tin)
    z = osf.osf_softmax_rows_ex(x, out_dtype=tout)
    check(z, oracle.softmax_masked(values(x)), f"{dtypes} T={T}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("Sq,heads", [(100, 3), (256, 2), (1000, 1)])
def test_causal_scaled_attention_weights(osf, dtype, Sq, heads):
    """Stacked [Sq, Sk=Sq] score matrices of several heads: row r keeps columns 0 .. r % Sq."""
    x32 = (si.normal_f32((heads * Sq, Sq), Sq, si.STREAM_X) * 11).astype(np.float32)
    x = to_dev(x32, dtype)
    scale = 64 ** -0.5
    z = osf.osf_softmax_rows_ex(x, scale=scale, causal_period=Sq)
    ref = oracle.softmax_masked(values(x), scale, Sq)
    check(z, ref, f"causal {dtype} Sq={Sq}")
    got = values(z)
    assert np.all(got[ref == 0] == 0), "masked columns must be exactly zero"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,T,period", [(2048, 2048, 2048), (3000, 2048, 1500), (500, 4096, 100000),
                                           (1000, 8192, 333)])
def test_causal_periods_long_rows(osf, dtype, rows, T, period):
    """Causal rows long enough that the rows keeping at most half their columns run with half the
    row buffer: whole and partial periods, a period longer than the rows, and one shorter than T."""
    x32 = (si.normal_f32((rows, T), rows + T, si.STREAM_X) * 9).astype(np.float32)
    x = to_dev(x32, dtype)
    z = osf.osf_softmax_rows_ex(x, scale=0.3, causal_period=period)
    ref = oracle.softmax_masked(values(x), 0.3, period)
    check(z, ref, f"causal {dtype} rows={rows} T={T} period={period}")
    assert np.all(values(z)[ref == 0] == 0), "masked columns must be exactly zero"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,T,period", [(1001, 1024, 333), (64, 512, 64), (7, 256, 8), (96, 128, 96)])
def test_causal_row_pairs(osf, dtype, rows, T, period):
    """Short causal rows (P <= T) run two complementary rows of a score matrix per CTA: an odd
    period (the middle row alone), a last partial matrix (rows % P != 0, partners past the end),
    fewer rows than one period, and in place."""
    x32 = (si.normal_f32((rows, T), rows * 7 + T, si.STREAM_X) * 9).astype(np.float32)
    x = to_dev(x32, dtype)
    ref = oracle.softmax_masked(values(x), 0.7, period)
    z = osf.osf_softmax_rows_ex(x, scale=0.7, causal_period=period)
    check(z, ref, f"pairs {dtype} rows={rows} T={T} period={period}")
    assert np.all(values(z)[ref == 0] == 0), "masked columns must be exactly zero"
    w = osf.osf_softmax_rows_ex(x, x, scale=0.7, causal_period=period)   # in place
    check(w, ref, f"pairs in place {dtype}")


def test_causal_bf16_full_size(osf):
    """The causal attention-weight workload (8 heads x [4096, 4096] bf16, scale 128^-0.5) as the
    benchmark runs it: every row against the oracle, in blocks of rows."""
    rows, T = 8 * 4096, 4096
    x = torch.from_numpy(si.softmax_rows_input(rows, T, seed=0)).cuda().to(torch.bfloat16)
    z = osf.osf_softmax_rows_ex(x, scale=128 ** -0.5, causal_period=4096)
    for r0 in range(0, rows, 4096):
        ref = oracle.softmax_masked(values(x[r0:r0 + 4096]), 128 ** -0.5, 4096)
        check(z[r0:r0 + 4096], ref, f"causal bf16 8x4096x4096 head {r0 // 4096}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_padded_row_strides_and_in_place(osf, dtype):
    x32 = si.softmax_rows_input(40, 1000, seed=5)
    x = to_dev(x32, dtype, pad=24)          # row stride 1024: aligned
    y = to_dev(x32, dtype, pad=3)           # row stride 1003: not 16-byte aligned
    ref = oracle.softmax_masked(values(x), 0.5, 0)
    zbuf = torch.full((40, 1000 + 8), 7.0, dtype=dtype, device="cuda")
    z = osf.osf_softmax_rows_ex(x, zbuf[:, :1000], scale=0.5)
    check(z, ref, f"strided {dtype}")
    assert torch.all(zbuf[:, 1000:] == 7.0), "padding of z written"
    check(osf.osf_softmax_rows_ex(y, scale=0.5), ref, f"unaligned {dtype}")
    w = osf.osf_softmax_rows_ex(y, y, scale=0.5)   # in place
    check(w, ref, f"in place {dtype}")


def test_bf16_rows_full_size(osf):
    """The softmax workload shape (4096 x 32768) in bf16 in and out, as the benchmark runs it:
    every row against the oracle (compared in blocks of rows to bound host memory)."""
    rows, T = 4096, 32768
    x = torch.from_numpy(si.softmax_rows_input(rows, T, seed=0)).cuda().to(torch.bfloat16)
    z = osf.osf_softmax_rows_ex(x)
    for r0 in range(0, rows, 512):
        check(z[r0:r0 + 512], oracle.softmax_masked(values(x[r0:r0 + 512])), f"bf16 4096x32768 rows {r0}+")


def test_long_rows_after_shorter_ones(osf):
    """Row lengths whose shared-memory needs differ, in the order long, short, long: the kernels'
    dynamic shared-memory limit is only ever raised, so the second long call still launches."""
    for T in (32768, 16384, 32768):
        x32 = si.softmax_rows_input(5, T, seed=T + 1)
        x = to_dev(x32, torch.bfloat16)
        check(osf.osf_softmax_rows_ex(x), oracle.softmax_masked(values(x)), f"bf16 T={T}")


@pytest.mark.parametrize("dtype,T,rows,period", [(torch.bfloat16, 17000, 1000, 1000), (torch.bfloat16, 20000, 6, 0),
                                                 (torch.float32, 16384, 9, 0), (torch.float32, 12000, 700, 700)])
def test_rows_half_shared_half_registers(osf, dtype, T, rows, period):
    """Rows of 32-64 KB keep their first part in shared memory and the rest in registers: causal
    limits before, at and after the split column, and whole rows."""
    x32 = (si.normal_f32((rows, T), rows + T, si.STREAM_X) * 7).astype(np.float32)
    x = to_dev(x32, dtype)
    z = osf.osf_softmax_rows_ex(x, scale=0.9, causal_period=period)
    ref = oracle.softmax_masked(values(x), 0.9, period)
    check(z, ref, f"split {dtype} T={T} rows={rows} period={period}")
    if period:
        assert np.all(values(z)[ref == 0] == 0), "masked columns must be exactly zero"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,T,period", [(64, 2048, 64), (33, 1000, 0), (12, 6000, 0), (5, 12000, 0),
                                           (4, 20000, 0), (3, 32768, 0)])
def test_negative_scale(osf, dtype, rows, T, period):
    """A negative scale is applied as |scale| to the values with their signs flipped on load; every
    staged path (paired causal rows, one CTA of 64, 128 or 256 threads, half in registers)."""
    x32 = (si.normal_f32((rows, T), rows * 3 + T, si.STREAM_X) * 5).astype(np.float32)
    x = to_dev(x32, dtype)
    z = osf.osf_softmax_rows_ex(x, scale=-0.6, causal_period=period)
    check(z, oracle.softmax_masked(values(x), -0.6, period), f"negative scale {dtype} T={T} period={period}")


@pytest.mark.parametrize("dtype,T", [(torch.bfloat16, 32768), (torch.float32, 16384), (torch.bfloat16, 4096)])
def test_long_rows_strided_and_in_place(osf, dtype, T):
    """Rows with a padded row stride (x and z strides differ) and in place, on the half-register
    path (32-64 KB rows) and on the paired causal path."""
    rows = 6
    x32 = (si.normal_f32((rows, T), T + 11, si.STREAM_X) * 6).astype(np.float32)
    x = to_dev(x32, dtype, pad=64)                        # row stride T + 64
    period = rows if T == 4096 else 0
    ref = oracle.softmax_masked(values(x), 1.3, period)
    zbuf = torch.full((rows, T + 128), 5.0, dtype=dtype, device="cuda")
    z = osf.osf_softmax_rows_ex(x, zbuf[:, :T], scale=1.3, causal_period=period)
    check(z, ref, f"strided {dtype} T={T}")
    assert torch.all(zbuf[:, T:] == 5.0), "padding of z written"
    w = osf.osf_softmax_rows_ex(x, x, scale=1.3, causal_period=period)   # in place
    check(w, ref, f"in place {dtype} T={T}")
