"""GPU parity of the few-rows float32 attention kernel against the oracle.

Float32 problems with at most 2048 query rows in all, at most 256 keys and D <= 64 run one warp
per query row, with the kv head's whole K and V staged in shared memory first ("softmax_attention",
section "实现思路": one program per query, keys in blocks, the running max / rescale / sum /
numerator recurrence).  Covered here: the `solve` shapes around the M = 64, N = 100, d = 32
workload, the largest staged key count (256) and the first one past it (257, the tiled kernel),
D not a multiple of 4 and rows whose pitch is not a 16-byte multiple (4-byte copies), GQA, the
top-left and bottom-right masks with Sq != Sk (rows that see no key: O = 0, lse = -inf), and
[B, S, H, D] views.  Tolerance: max abs 1e-4, the float32 bar.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_f32_close, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("M,N,d", [(64, 100, 32), (1, 1, 1), (4, 256, 64), (63, 64, 16), (5, 65, 20),
                                   (2048, 7, 8), (64, 257, 32), (3, 192, 63)])
def test_solve_shapes(osf, M, N, d):
    Q, K, V = si.qkv((M, d), (N, d), seed=M * 7 + N * 3 + d)
    out = torch.full((M, d), 7.0, device="cuda")
    osf.osf_attn_fwd(f32_tensor(Q), f32_tensor(K), f32_tensor(V), out, M, N, d)
    ref, _ = oracle.attention(Q, K, V)
    assert_f32_close(out.cpu().numpy(), ref, atol=1e-4, what=f"solve {M}x{N}x{d}")


def on_device(a, layout, pad):
    t = f32_tensor(a)
    B, H, S, D = t.shape
    if layout == "bshd":
        store = torch.zeros((B, S, H, D + pad), device="cuda")
        store[..., :D] = t.permute(0, 2, 1, 3)
        return store[..., :D].transpose(1, 2)
    store = torch.zeros((B, H, S, D + pad), device="cuda")
    store[..., :D] = t
    return store[..., :D]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,mask,layout,pad", [
    (2, 4, 2, 17, 200, 32, "top_left", "bhsd", 0),
    (1, 6, 3, 40, 23, 48, "bottom_right", "bshd", 0),     # 17 rows see no key
    (3, 2, 1, 9, 256, 40, "none", "bshd", 0),
    (1, 4, 4, 33, 257, 32, "top_left", "bhsd", 0),       # past the staged key count
    (1, 2, 1, 50, 120, 20, "bottom_right", "bhsd", 1),   # odd row pitch: 4-byte copies
    (2, 8, 2, 1, 250, 64, "none", "bshd", 0),            # one row per head
])
def test_gqa_masks_and_views(osf, B, Hq, Hkv, Sq, Sk, D, mask, layout, pad):
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=B + 5 * Sq + 11 * Sk + D)
    Q, K, V = (on_device(a, layout, pad) for a in (q, k, v))
    out = torch.full((B, Hq, Sq, D), 3.0, device="cuda")
    lse = torch.empty(B, Hq, Sq, device="cuda")
    osf.osf_attn_fwd_gqa_ex(Q, K, V, out=out, mask=mask, lse=lse)
    ref, ref_lse = oracle.attention_gqa(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), mask=mask)
    what = f"{B},{Hq},{Hkv},{Sq},{Sk},{D} {mask} {layout} pad={pad}"
    assert_f32_close(out.cpu().numpy(), ref, atol=1e-4, what=what)
    got_lse = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), what + " lse -inf rows"
    fin = np.isfinite(ref_lse)
    assert_f32_close(got_lse[fin], ref_lse[fin], atol=1e-4, what=what + " lse")


def test_solve_is_deterministic(osf):
    Q, K, V = (f32_tensor(a) for a in si.qkv((64, 32), (100, 32), seed=0))
    a, b = torch.empty(64, 32, device="cuda"), torch.empty(64, 32, device="cuda")
    osf.osf_attn_fwd(Q, K, V, a, 64, 100, 32)
    osf.osf_attn_fwd(Q, K, V, b, 64, 100, 32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_large_scores_and_scale_override(osf, causal):
    """Scores of a few hundred (Q scaled by 30) and an explicit scale: the running maximum keeps
    every exponent <= 0 and the per-block rescale stays exact in float32."""
    B, Hq, Hkv, S, D = 1, 4, 2, 150, 32
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=77 + causal)
    q = (q * 30.0).astype(np.float32)
    scale = 0.3
    lse = torch.empty(B, Hq, S, device="cuda")
    o = osf.osf_attn_fwd_gqa(f32_tensor(q), f32_tensor(k), f32_tensor(v), causal=causal, scale=scale, lse=lse)
    ref, ref_lse = oracle.attention_gqa(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                                        causal=causal, scale=scale)
    assert_f32_close(o.cpu().numpy(), ref, atol=1e-4, what=f"large scores causal={causal}")
    assert_f32_close(lse.cpu().numpy(), ref_lse, atol=1e-3, what="lse")
