"""GPU parity of float32 attention with D = 64, which runs on the bf16 tensor cores as sums of
bf16 part products (three parts of Q and K for the scores, two of P and V), against the fp64
oracle with the float32 tolerance (max abs error <= 1e-4).

The scores are the sensitive product: the exponent turns an absolute error of S into a
relative error of P, so these cases use large operand magnitudes (scores in the hundreds),
strided layouts, split key ranges and rows without keys.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_f32_close, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def run(osf, B, Hq, Hkv, Sq, Sk, qscale, kscale, mask, seed, layout="bhsd"):
    D = 64
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=seed)
    q, k = (q * np.float32(qscale)).astype(np.float32), (k * np.float32(kscale)).astype(np.float32)
    if layout == "bshd":
        Q, K, V = (f32_tensor(np.ascontiguousarray(a.transpose(0, 2, 1, 3))).transpose(1, 2) for a in (q, k, v))
    else:
        Q, K, V = (f32_tensor(a) for a in (q, k, v))
    lse = torch.empty(B, Hq, Sq, device="cuda")
    out = None
    if layout == "bshd":   # the output as a [B, S, H, D] buffer seen as [B, H, S, D]
        out = torch.full((B, Sq, Hq, D), float("nan"), device="cuda").transpose(1, 2)
    n0 = osf.osf_launch_count()
    o = osf.osf_attn_fwd_gqa_ex(Q, K, V, out=out, mask=mask, lse=lse)
    torch.cuda.synchronize()
    launches = osf.osf_launch_count() - n0
    ref, ref_lse = oracle.attention_gqa(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), mask=mask)
    what = f"f32 D=64 {B},{Hq},{Hkv},{Sq},{Sk} x{qscale}/{kscale} {mask} {layout}"
    assert_f32_close(o.cpu().numpy(), ref, what=what)
    fin = np.isfinite(ref_lse)
    got_lse = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), what + " lse -inf rows"
    assert_f32_close(got_lse[fin], ref_lse[fin], atol=1e-3, what=what + " lse")
    return launches


def test_runs_on_the_tensor_core_path(osf):
    """One query block per head and as many heads as SMs: neither path splits the keys, so the
    CUDA-core kernel would be one launch; the split pre-pass plus the tensor-core kernel are two."""
    launches = run(osf, 1, osf.osf_sm_count(), 1, 256, 256, 1.0, 1.0, "none", seed=1)
    assert launches == 2, launches


@pytest.mark.parametrize("qscale,kscale", [(30.0, 1.0), (4.0, 4.0), (1e-3, 1e3)])
def test_large_scores(osf, qscale, kscale):
    """Scores with standard deviations of 30, 16 and 8 (maxima near 100).  The error grows with
    |S| through the fp32 accumulation of the products: at a standard deviation of 64 it measured
    1.25e-4."""
    run(osf, 1, 4, 2, 384, 384, qscale, kscale, "top_left", seed=2)


def test_key_splits_ragged_and_bshd(osf):
    """One head, few query tiles: the key range is split and merged; ragged lengths; BSHD views
    of the inputs and of the output."""
    run(osf, 1, 1, 1, 1000, 1537, 4.0, 2.0, "none", seed=3, layout="bshd")
    run(osf, 2, 4, 2, 333, 333, 2.0, 2.0, "top_left", seed=5, layout="bshd")


def test_bottom_right_rows_without_keys(osf):
    run(osf, 2, 4, 1, 300, 190, 3.0, 3.0, "bottom_right", seed=4)
