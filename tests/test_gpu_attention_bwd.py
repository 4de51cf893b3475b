"""GPU parity of ``osf_attn_bwd_gqa`` (dQ, dK, dV) against ``oracle.attention_gqa_bwd``.

The forward pass runs on the GPU (``osf_attn_fwd_gqa_ex``) to produce O and lse, as a training
step would; the oracle recomputes everything in fp64 from Q, K, V, dO.

Tolerances.  bf16: the gradients are sums of products whose factors P and dS are rounded to
bf16 (2^-9 relative) before the tensor-core products, and the results are rounded to bf16;
the error therefore scales with the size of the terms, i.e. with the tensor's largest
gradient, not with each element: |gpu - ref| <= 2e-2 * max|ref| + 1e-2 * |ref| (the forward's
bf16 pair, scaled; about 4x the worst error seen).  float32 (CUDA-core path, fp32 throughout):
|gpu - ref| <= 1e-4 * max(1, max|ref|).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import bf16_tensor, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def f64(a, dtype):
    return si.bf16_bits_to_f32(a).astype(np.float64) if dtype == "bf16" else a.astype(np.float64)


def check_grad(got, ref, dtype, what):
    g = got.float().cpu().numpy()
    scale = np.abs(ref).max() if ref.size else 0.0
    err = np.abs(g - ref)
    if dtype == "bf16":
        bound = 2e-2 * scale + 1e-2 * np.abs(ref)
    else:
        bound = 1e-4 * max(1.0, scale) + 0 * ref
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} off, worst err {err.max():.3g} (max|ref| {scale:.3g})"
    assert np.isfinite(g).all(), what + " not finite"


def rowsum_only_workspace(B, Hq, Sq):
    """A workspace with room for the row sums alone: the tensor-core path then recomputes S and
    dP for dQ instead of storing dS."""
    return torch.empty((B * Hq * Sq * 4 + 255) // 256 * 256, dtype=torch.uint8, device="cuda")


def run(osf, B, Hq, Hkv, Sq, Sk, D, dtype, mask, seed=0, store_ds=True):
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=seed, dtype=dtype)
    g = si.qkv((B, Hq, Sq, D), (1, 1, 1, D), seed=seed + 1000, dtype=dtype)[0]
    dev = bf16_tensor if dtype == "bf16" else f32_tensor
    Q, K, V, G = dev(q), dev(k), dev(v), dev(g)
    lse = torch.empty(B, Hq, Sq, device="cuda")
    O = osf.osf_attn_fwd_gqa_ex(Q, K, V, mask=mask, lse=lse)
    ws = None if store_ds else rowsum_only_workspace(B, Hq, Sq)
    dq, dk, dv = osf.osf_attn_bwd_gqa(Q, K, V, O, G, lse, mask=mask, workspace=ws)
    rq, rk, rv = oracle.attention_gqa_bwd(f64(q, dtype), f64(k, dtype), f64(v, dtype), f64(g, dtype), mask=mask)
    what = f"{dtype} {B},{Hq},{Hkv},{Sq},{Sk},{D} {mask} store_ds={store_ds}"
    check_grad(dq, rq, dtype, what + " dq")
    check_grad(dk, rk, dtype, what + " dk")
    check_grad(dv, rv, dtype, what + " dv")


@pytest.mark.parametrize("store_ds", [True, False])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask", ["none", "top_left", "bottom_right"])
def test_bf16_tensor_core_backward(osf, D, mask, store_ds):
    """Both tensor-core paths: dS stored and dQ as one product over it (the default workspace),
    and dQ recomputing S and dP (a workspace of row sums only)."""
    Sk = 333 if mask == "bottom_right" else 200
    run(osf, 1, 4, 2, 200, Sk, D, "bf16", mask, seed=D, store_ds=store_ds)


@pytest.mark.parametrize("mask", ["none", "top_left", "bottom_right"])
def test_f32_backward(osf, mask):
    run(osf, 1, 4, 2, 100, 130 if mask == "bottom_right" else 100, 64, "f32", mask, seed=7)


@pytest.mark.parametrize("D", [32, 96])
def test_bf16_other_head_dims_backward(osf, D):
    run(osf, 2, 4, 4, 77, 77, D, "bf16", "top_left", seed=D)


@pytest.mark.parametrize("store_ds", [True, False])
def test_backward_ragged_multi_block_gqa(osf, store_ds):
    """Several key and query blocks with ragged ends, G = 4 and G = 3 (the dQ product pairs the
    query heads of a group when G is even), bottom-right with Sq > Sk (rows without keys must send
    back nothing), and more query tiles than SMs hold items at once."""
    run(osf, 2, 8, 2, 300, 190, 128, "bf16", "bottom_right", seed=11, store_ds=store_ds)
    run(osf, 1, 8, 2, 1000, 1000, 64, "bf16", "top_left", seed=12, store_ds=store_ds)
    run(osf, 3, 16, 4, 1100, 700, 128, "bf16", "none", seed=13, store_ds=store_ds)
    run(osf, 1, 6, 2, 260, 300, 64, "bf16", "top_left", seed=14, store_ds=store_ds)   # odd group size


def test_backward_paths_agree_and_repeat(osf):
    """The stored-dS path and the recomputing path give the same dK and dV bit for bit (the dK/dV
    CTAs are the same; storing dS only adds writes) and dQ within bf16 rounding of each other; each
    path repeats its own result exactly."""
    B, Hq, Hkv, S, D = 1, 8, 2, 700, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=21, dtype="bf16")
    g = si.qkv((B, Hq, S, D), (1, 1, 1, D), seed=1021, dtype="bf16")[0]
    Q, K, V, G = (bf16_tensor(a) for a in (q, k, v, g))
    lse = torch.empty(B, Hq, S, device="cuda")
    O = osf.osf_attn_fwd_gqa_ex(Q, K, V, mask="top_left", lse=lse)
    a = osf.osf_attn_bwd_gqa(Q, K, V, O, G, lse, mask="top_left")
    a2 = osf.osf_attn_bwd_gqa(Q, K, V, O, G, lse, mask="top_left")
    small = rowsum_only_workspace(B, Hq, S)
    r = osf.osf_attn_bwd_gqa(Q, K, V, O, G, lse, mask="top_left", workspace=small)
    r2 = osf.osf_attn_bwd_gqa(Q, K, V, O, G, lse, mask="top_left", workspace=small)
    torch.cuda.synchronize()
    for x, y in zip(a, a2):
        assert torch.equal(x, y)
    for x, y in zip(r, r2):
        assert torch.equal(x, y)
    assert torch.equal(a[1], r[1]) and torch.equal(a[2], r[2])
    d = (a[0].float() - r[0].float()).abs().max().item()
    assert d <= 2e-2 * r[0].float().abs().max().item(), d


def test_backward_rejects_overlaps_and_missing_workspace(osf):
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 8, device="cuda")
    lib = osf.lib()
    assert lib.osf_attn_bwd_gqa(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                lse.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), osf.OSF_BF16, 1, 2, 2, 8,
                                8, 64, 0, 0.0, None, 0, None) == osf.OSF_ERR_INVALID
    out = [torch.empty_like(q) for _ in range(3)]
    assert lib.osf_attn_bwd_gqa(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                lse.data_ptr(), *(t.data_ptr() for t in out), osf.OSF_BF16, 1, 2, 2, 8, 8, 64, 0,
                                0.0, None, 0, None) == osf.OSF_ERR_WORKSPACE


def test_backward_full_size(osf):
    """The benchmark's backward (B=2, Hq=32, Hkv=8, S=4096, D=128, causal) in its own launch
    configuration, every element against the oracle, one kv group at a time (a group's dQ, dK and
    dV depend only on its own Q, K, V and dO)."""
    B, Hq, Hkv, S, D = 2, 32, 8, 4096, 128
    G = Hq // Hkv
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=5, dtype="bf16")
    g = si.qkv((B, Hq, S, D), (1, 1, 1, D), seed=1005, dtype="bf16")[0]
    Q, K, V, GO = (bf16_tensor(a) for a in (q, k, v, g))
    lse = torch.empty(B, Hq, S, device="cuda")
    O = osf.osf_attn_fwd_gqa_ex(Q, K, V, mask="top_left", lse=lse)
    dq, dk, dv = osf.osf_attn_bwd_gqa(Q, K, V, O, GO, lse, mask="top_left")
    torch.cuda.synchronize()
    for b, kvh in ((b, h) for b in range(B) for h in range(Hkv)):
        hs = slice(kvh * G, (kvh + 1) * G)
        rq, rk, rv = oracle.attention_gqa_bwd(f64(q[b:b + 1, hs], "bf16"), f64(k[b:b + 1, kvh:kvh + 1], "bf16"),
                                              f64(v[b:b + 1, kvh:kvh + 1], "bf16"), f64(g[b:b + 1, hs], "bf16"),
                                              mask="top_left")
        what = f"full size b={b} kv head {kvh}"
        check_grad(dq[b:b + 1, hs], rq, "bf16", what + " dq")
        check_grad(dk[b:b + 1, kvh:kvh + 1], rk, "bf16", what + " dk")
        check_grad(dv[b:b + 1, kvh:kvh + 1], rv, "bf16", what + " dv")


@pytest.mark.parametrize("store_ds", [True, False])
def test_backward_rows_with_very_negative_scores_and_a_ragged_key_tail(osf, store_ds):
    """Every score of every row far below zero (Q and K pointing apart, scale 10) with Sk not a
    multiple of 128: lse is near -370, so e^-lse overflows float32 for the zero-filled key rows
    past Sk, and those rows must not reach dQ.  The gradients stay finite and match the oracle.
    (The K offset is kept to about the spread of K: with a large common offset the bf16 rounding of
    dS alone, amplified by |K|, reaches the bf16 bound in dQ whatever the kernel.)"""
    B, Hq, Hkv, Sq, Sk, D, scale = 1, 4, 2, 150, 190, 64, 10.0
    k = np.abs(si.normal_f32((B, Hkv, Sk, D), 31, si.STREAM_K)) * np.float32(0.5) + np.float32(0.5)
    q = -np.abs(si.normal_f32((B, Hq, Sq, D), 31, si.STREAM_Q)) * np.float32(0.5) - np.float32(0.5)
    v = si.normal_f32((B, Hkv, Sk, D), 31, si.STREAM_V)
    g = si.normal_f32((B, Hq, Sq, D), 32, si.STREAM_V)
    qb, kb, vb, gb = (si.f32_to_bf16_bits(a) for a in (q, k, v, g))
    Q, K, V, G = (bf16_tensor(a) for a in (qb, kb, vb, gb))
    lse = torch.empty(B, Hq, Sq, device="cuda")
    O = osf.osf_attn_fwd_gqa_ex(Q, K, V, mask="none", scale=scale, lse=lse)
    assert float(lse.max()) < -100.0   # e^100 is past the float32 range
    ws = None if store_ds else rowsum_only_workspace(B, Hq, Sq)
    dq, dk, dv = osf.osf_attn_bwd_gqa(Q, K, V, O, G, lse, mask="none", scale=scale, workspace=ws)
    rq, rk, rv = oracle.attention_gqa_bwd(f64(qb, "bf16"), f64(kb, "bf16"), f64(vb, "bf16"), f64(gb, "bf16"),
                                          mask="none", scale=scale)
    what = f"very negative scores store_ds={store_ds}"
    check_grad(dq, rq, "bf16", what + " dq")
    check_grad(dk, rk, "bf16", what + " dk")
    check_grad(dv, rv, "bf16", what + " dv")
