"""GPU parity of ``osf_attn_fwd_gqa_ex``: strided views and the mask modes, against the oracle.

[Q3] "stride的作用": a head split or a transpose of any but the last dimension only changes
strides, and a broadcast dimension has stride 0.  The GPU reads each layout in place; the oracle
sees the same logical [B, H, S, D] values.  Masks: ``top_left`` (the pages' tril(ones(Sq, Sk)))
and ``bottom_right`` (row i sees keys up to i + Sk - Sq; a reading, not on the pages) for any
Sq, Sk, including rows that see no key (O = 0, lse = -inf).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_bf16_close, assert_f32_close, bf16_tensor, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def logical(bits, dtype):
    return si.bf16_bits_to_f32(bits).astype(np.float64) if dtype == "bf16" else bits.astype(np.float64)


def on_device(bits, dtype, layout="bhsd", pad=0):
    """Logical [B, H, S, D] view of the values, stored as `layout` (bhsd or bshd), with `pad`
    unused elements after each row of D."""
    t = bf16_tensor(bits) if dtype == "bf16" else f32_tensor(bits)
    B, H, S, D = t.shape
    if layout == "bshd":
        store = torch.zeros((B, S, H, D + pad), dtype=t.dtype, device=t.device)
        store[..., :D] = t.permute(0, 2, 1, 3)
        return store[..., :D].transpose(1, 2)
    store = torch.zeros((B, H, S, D + pad), dtype=t.dtype, device=t.device)
    store[..., :D] = t
    return store[..., :D]


def check(got, ref, dtype, what):
    g = got.float().cpu().numpy()
    return assert_bf16_close(g, ref, what) if dtype == "bf16" else assert_f32_close(g, ref, what=what)


def run(osf, B, Hq, Hkv, Sq, Sk, D, dtype, mask, layout="bhsd", out_layout="bhsd", pad=0, seed=0):
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=seed, dtype=dtype)
    Q, K, V = (on_device(a, dtype, layout, pad) for a in (q, k, v))
    out = on_device(np.zeros((B, Hq, Sq, D), dtype=q.dtype), dtype, out_layout)
    lse = torch.empty(B, Hq, Sq, device="cuda")
    osf.osf_attn_fwd_gqa_ex(Q, K, V, out=out, mask=mask, lse=lse)
    ref, ref_lse = oracle.attention_gqa(logical(q, dtype), logical(k, dtype), logical(v, dtype), mask=mask)
    what = f"{dtype} {layout}->{out_layout} pad={pad} {B},{Hq},{Hkv},{Sq},{Sk},{D} {mask}"
    check(out, ref, dtype, what)
    got_lse = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), what + " lse -inf rows"
    fin = np.isfinite(ref_lse)
    assert_f32_close(got_lse[fin], ref_lse[fin], atol=1e-3, what=what + " lse")
    return out, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask", ["none", "top_left"])
def test_bshd_views_on_the_tensor_core_path(osf, D, mask):
    run(osf, 2, 8, 2, 300, 300, D, "bf16", mask, layout="bshd", out_layout="bshd", seed=D)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("Sq,Sk", [(200, 700), (130, 129), (700, 200), (1, 333), (5, 1000)])
@pytest.mark.parametrize("mask", ["top_left", "bottom_right"])
def test_masks_with_unequal_lengths(osf, dtype, Sq, Sk, mask):
    D = 128 if dtype == "bf16" else 64
    run(osf, 1, 4, 2, Sq, Sk, D, dtype, mask, layout="bshd", seed=Sq + 3 * Sk)


def test_bottom_right_chunked_prefill_bf16_d64(osf):
    """A chunk of 256 new rows after a 1536-key cache, [B, S, H, D] layout."""
    run(osf, 2, 8, 4, 256, 1792, 64, "bf16", "bottom_right", layout="bshd", out_layout="bshd", seed=17)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_from_a_bshd_cache(osf, dtype):
    run(osf, 3, 8, 2, 1, 4099, 128, dtype, "bottom_right", layout="bshd", out_layout="bshd", seed=19)


def test_unaligned_row_pitch_falls_back_and_stays_correct(osf):
    """Rows padded by 3 elements: strides are not 16-byte multiples, so no TMA path applies."""
    run(osf, 1, 4, 2, 200, 200, 64, "bf16", "top_left", pad=3, seed=23)
    run(osf, 1, 4, 2, 1, 500, 128, "bf16", "none", pad=3, seed=24)


def test_broadcast_kv_heads_with_stride_zero(osf):
    """One kv head expanded over 4 heads (stride 0) equals the same kv head stored 4 times."""
    B, Hq, Sq, Sk, D = 1, 8, 200, 200, 128
    q, k, v = si.qkv((B, Hq, Sq, D), (B, 1, Sk, D), seed=29, dtype="bf16")
    Q = bf16_tensor(q)
    K1, V1 = bf16_tensor(k), bf16_tensor(v)
    Ke, Ve = K1.expand(B, 4, Sk, D), V1.expand(B, 4, Sk, D)
    assert Ke.stride(1) == 0
    out = osf.osf_attn_fwd_gqa_ex(Q, Ke, Ve, mask="top_left")
    ref, _ = oracle.attention_gqa(logical(q, "bf16"), logical(k, "bf16"), logical(v, "bf16"), mask="top_left")
    check(out, ref, "bf16", "broadcast kv heads")


def test_full_size_workload_in_bshd_layout_sampled(osf):
    """The GQA causal prefill workload (B=2, Hq=32, Hkv=8, S=4096, D=128) stored [B, S, H, D],
    checked at sampled rows; it must also equal the contiguous call exactly."""
    B, Hq, Hkv, S, D = 2, 32, 8, 4096, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=0, dtype="bf16")
    Q, K, V = (on_device(a, "bf16", "bshd") for a in (q, k, v))
    out = on_device(np.zeros((B, Hq, S, D), dtype=q.dtype), "bf16", "bshd")
    osf.osf_attn_fwd_gqa_ex(Q, K, V, out=out, mask="top_left")
    contiguous = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out, contiguous), "strided and contiguous calls differ"
    rng = np.random.default_rng(1)
    rows = [(b, h, i) for b in range(B) for h in range(0, Hq, 5) for i in (0, 255, 256, S - 1, int(rng.integers(0, S)))]
    ref, _ = oracle.attention_rows(logical(q, "bf16"), logical(k, "bf16"), logical(v, "bf16"), rows, mask="top_left")
    of = out.float().cpu().numpy()
    assert_bf16_close(np.stack([of[b, h, i] for b, h, i in rows]), ref, "bshd full size")


def test_bottom_right_rows_without_keys_no_key_split(osf):
    """More work items than SMs (no key split): the first Sq - Sk rows see no key."""
    out, _ = run(osf, 2, 80, 8, 700, 200, 64, "bf16", "bottom_right", layout="bshd", seed=31)
    assert torch.all(out[:, :, :500] == 0)


@pytest.mark.parametrize("Sq,mask", [(2, "bottom_right"), (4, "bottom_right"), (3, "top_left"), (4, "none")])
def test_speculative_rows_on_the_decode_kernel(osf, Sq, mask):
    """G * Sq <= 16 query rows per kv head (here G = 4): the decode kernel with per-row limits."""
    run(osf, 2, 16, 4, Sq, 5003, 128, "bf16", mask, layout="bshd", seed=41 + Sq)
    run(osf, 1, 8, 2, Sq, 700, 64, "bf16", mask, seed=43 + Sq)


def test_chunked_prefill_full_size(osf):
    """The chunked-prefill workload at full size (1024 new rows after a 3072-key cache: B=2,
    Hq=32, Hkv=8, Sq=1024, Sk=4096, D=128, bottom-right), every element of O and lse."""
    run(osf, 2, 32, 8, 1024, 4096, 128, "bf16", "bottom_right", seed=53)


def test_speculative_decode_full_size(osf):
    """The speculative-decode workload at full size (4 draft rows per head against a 32768-key
    cache: B=8, Hq=32, Hkv=8, Sq=4, Sk=32768, D=128, bottom-right), every element of O and lse."""
    run(osf, 8, 32, 8, 4, 32768, 128, "bf16", "bottom_right", seed=59)
