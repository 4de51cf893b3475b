"""Key splits of the tensor-core forward, and how they are merged.

With fewer work items than SMs the key range is split.  When a query block's splits fit one
thread-block cluster (at most 8) they are merged inside the forward kernel through distributed
shared memory, so the forward is the only launch (after the float32 pre-pass); with more splits a
combine kernel merges the partial states.  Both routes are checked against the fp64 oracle,
with the log-sum-exp they return.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_bf16_close, assert_f32_close, bf16_tensor, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def run(osf, dtype, B, Hq, Hkv, Sq, Sk, D, mask, seed):
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=seed, dtype=dtype)
    dev = bf16_tensor if dtype == "bf16" else f32_tensor
    f64 = (lambda a: si.bf16_bits_to_f32(a).astype(np.float64)) if dtype == "bf16" else (lambda a: a.astype(np.float64))
    lse = torch.full((B, Hq, Sq), float("nan"), device="cuda")
    n0 = osf.osf_launch_count()
    o = osf.osf_attn_fwd_gqa_ex(dev(q), dev(k), dev(v), mask=mask, lse=lse)
    torch.cuda.synchronize()
    launches = osf.osf_launch_count() - n0
    ref, ref_lse = oracle.attention_gqa(f64(q), f64(k), f64(v), mask=mask)
    what = f"{dtype} {B},{Hq},{Hkv},{Sq},{Sk},{D} {mask}"
    got = o.float().cpu().numpy()
    if dtype == "bf16":
        assert_bf16_close(got, ref, what)
    else:
        assert_f32_close(got, ref, what=what)
    got_lse = lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), what + ": rows without keys"
    assert_f32_close(got_lse[fin], ref_lse[fin], atol=1e-3, what=what + " lse")
    return launches


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_head_4096(osf, dtype):
    """M = N = 4096, d = 64: 16 query blocks x 8 key splits.  Whether 16 clusters of 8 CTAs fit
    the GPU at once decides the route (on GB300 15 do, so the combine kernel merges)."""
    launches = run(osf, dtype, 1, 1, 1, 4096, 4096, 64, "none", seed=31)
    assert launches in ((1, 2) if dtype == "bf16" else (2, 3))


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_splits_merged_in_kernel(osf, D):
    """Three splits of three key tiles; the last query block has one ragged tile of rows."""
    assert run(osf, "bf16", 2, 4, 2, 333, 333, D, "top_left", seed=32) == 1


def test_causal_gqa_four_splits_merged_in_kernel(osf):
    """32 query blocks x 4 key splits: 32 clusters of 4."""
    assert run(osf, "bf16", 2, 4, 2, 1024, 1024, 128, "top_left", seed=35) == 1


def test_float32_splits_merged_in_kernel(osf):
    """float32 (bf16 parts on the tensor cores): the split pre-pass, then the merging forward."""
    assert run(osf, "f32", 1, 4, 2, 384, 384, 64, "top_left", seed=36) == 2


def test_bottom_right_splits_without_keys(osf):
    """Bottom-right causal with Sq > Sk: early rows see no key in any split (O = 0, lse = -inf)."""
    assert run(osf, "bf16", 1, 2, 1, 700, 500, 128, "bottom_right", seed=33) == 1


def test_many_splits_use_the_combine_kernel(osf):
    """One query block over 32 key tiles: 32 splits, more than a cluster holds."""
    assert run(osf, "bf16", 1, 1, 1, 256, 4096, 128, "none", seed=34) == 2
