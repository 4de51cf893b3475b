"""GPU parity of the attention paths against the fp64 oracle, through the C ABI binding.

Inputs are the seeded i.i.d. N(0, 1) draws of ``seeded_inputs``; bf16 cases feed the oracle
the exact bf16 values the GPU receives.  Sizes span several tiles plus ragged tails; the
full-size workloads are checked element by element where the oracle is quick (single head
4096 x 4096, decode) and at sampled rows otherwise (GQA causal prefill).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_bf16_close, assert_f32_close, bf16_tensor, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def f64(bits_or_f32, dtype):
    return si.bf16_bits_to_f32(bits_or_f32).astype(np.float64) if dtype == "bf16" \
        else bits_or_f32.astype(np.float64)


def dev(a, dtype):
    return bf16_tensor(a) if dtype == "bf16" else f32_tensor(a)


def check(got, ref, dtype, what):
    got = got.float().cpu().numpy() if hasattr(got, "cpu") else got
    return assert_bf16_close(got, ref, what) if dtype == "bf16" else assert_f32_close(got, ref, what=what)


# ------------------------------------------------------------- single head (attn_fwd)
def test_attn_fwd_tail_block_m64_n100_d32(osf):
    """The first workload: M=64, N=100 (a ragged last key block), d=32, float32."""
    Q, K, V = si.qkv((64, 32), (100, 32), seed=0)
    out = torch.empty(64, 32, device="cuda")
    osf.solve(f32_tensor(Q), f32_tensor(K), f32_tensor(V), out, 64, 100, 32)
    ref, _ = oracle.attention(Q, K, V)
    check(out, ref, "f32", "attn_fwd 64x100x32")


@pytest.mark.parametrize("M", [1, 7, 31, 33, 100])
@pytest.mark.parametrize("N", [1, 7, 33, 100, 129])
@pytest.mark.parametrize("d", [1, 3, 32, 64, 100, 128, 200, 256])
def test_attn_fwd_small_shapes(osf, M, N, d):
    Q, K, V = si.qkv((M, d), (N, d), seed=M * 1000 + N * 10 + d)
    out = torch.empty(M, d, device="cuda")
    osf.osf_attn_fwd(f32_tensor(Q), f32_tensor(K), f32_tensor(V), out, M, N, d)
    torch.cuda.synchronize()
    ref, _ = oracle.attention(Q, K, V)
    check(out, ref, "f32", f"attn_fwd {M}x{N}x{d}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_head_4096_d64(osf, dtype):
    """The second workload: M = N = 4096, d = 64, float32 and the same draws cast to bf16."""
    Q, K, V = si.qkv((1, 1, 4096, 64), (1, 1, 4096, 64), seed=0, dtype=dtype)
    o = osf.osf_attn_fwd_gqa(dev(Q, dtype), dev(K, dtype), dev(V, dtype))
    ref, _ = oracle.attention(f64(Q, dtype)[0, 0], f64(K, dtype)[0, 0], f64(V, dtype)[0, 0])
    check(o[0, 0], ref, dtype, f"single head 4096 {dtype}")
    if dtype == "f32":
        out = torch.empty(4096, 64, device="cuda")
        osf.solve(f32_tensor(Q[0, 0]), f32_tensor(K[0, 0]), f32_tensor(V[0, 0]), out, 4096, 4096, 64)
        check(out, ref, dtype, "solve 4096")


# ------------------------------------------------------------------ batched GQA prefill
GQA_SMALL = [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 4, 2, 300, 300, 128, True),
    (2, 8, 2, 257, 257, 128, True),
    (1, 4, 4, 130, 130, 64, True),
    (2, 4, 1, 200, 333, 64, False),
    (1, 8, 8, 129, 129, 128, False),
    (1, 2, 1, 1000, 1000, 128, True),
    (1, 2, 2, 64, 500, 96, False),
    (3, 6, 3, 17, 17, 32, True),
    (1, 2, 1, 5, 3, 128, False),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", GQA_SMALL)
def test_gqa_small(osf, dtype, B, Hq, Hkv, Sq, Sk, D, causal):
    seed = B + 7 * Hq + 31 * Sq + D
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=seed, dtype=dtype)
    lse = torch.empty(B, Hq, Sq, device="cuda")
    o = osf.osf_attn_fwd_gqa(dev(q, dtype), dev(k, dtype), dev(v, dtype), causal=causal, lse=lse)
    ref, ref_lse = oracle.attention_gqa(f64(q, dtype), f64(k, dtype), f64(v, dtype), causal=causal)
    check(o, ref, dtype, f"gqa {dtype} {B},{Hq},{Hkv},{Sq},{Sk},{D},c={causal}")
    assert_f32_close(lse.cpu().numpy(), ref_lse, atol=1e-3, what="lse")


def test_gqa_causal_prefill_full_size(osf):
    """The GQA causal prefill workload at full size (B=2, Hq=32, Hkv=8, S=4096, D=128, bf16), in
    the launch configuration the benchmark times: every output element and every lse against the
    oracle (64 heads of explicit 4096 x 4096 fp64 scores), and two calls bit-identical."""
    B, Hq, Hkv, S, D = 2, 32, 8, 4096, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=0, dtype="bf16")
    lse = torch.empty(B, Hq, S, device="cuda")
    o = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=True, lse=lse)
    o2 = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2), "two identical calls differ"
    ref, ref_lse = oracle.attention_gqa(*(si.bf16_bits_to_f32(a) for a in (q, k, v)), causal=True)
    assert_bf16_close(o.float().cpu().numpy(), ref, "gqa prefill full size, every element")
    assert_f32_close(lse.cpu().numpy(), ref_lse, atol=1e-3, what="lse, every row")


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_more_items_than_sms(osf, causal):
    """More (b, head, 256-row block) work items than SMs, with a ragged last block: each CTA
    of the tensor-core prefill walks several items and carries its pipeline across them."""
    B, Hq, Hkv, S, D = 2, 40, 8, 1000, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=21 + causal, dtype="bf16")
    lse = torch.empty(B, Hq, S, device="cuda")
    o = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=causal, lse=lse)
    ref, ref_lse = oracle.attention_gqa(*(si.bf16_bits_to_f32(a) for a in (q, k, v)), causal=causal)
    check(o, ref, "bf16", f"gqa many items causal={causal}")
    assert_f32_close(lse.cpu().numpy(), ref_lse, atol=1e-3, what="lse")


def test_output_16_byte_aligned_only(osf):
    """An output that starts 16 bytes past a 32-byte boundary takes the 16-byte store path."""
    B, Hq, Hkv, S, D = 1, 4, 2, 300, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=23, dtype="bf16")
    n = B * Hq * S * D
    out = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")[8:].view(B, Hq, S, D)
    assert out.data_ptr() % 32 == 16
    osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), out=out, causal=True)
    ref, _ = oracle.attention_gqa(*(si.bf16_bits_to_f32(a) for a in (q, k, v)), causal=True)
    check(out, ref, "bf16", "16-byte aligned output")


# ----------------------------------------------------------------------------- decode
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_decode_split_invariance(osf, dtype, splits):
    B, Hq, Hkv, Sk, D = 2, 8, 2, 3001, 128
    q, k, v = si.qkv((B, Hq, 1, D), (B, Hkv, Sk, D), seed=5, dtype=dtype)
    lse = torch.empty(B, Hq, 1, device="cuda")
    o = osf.osf_attn_decode_gqa(dev(q, dtype), dev(k, dtype), dev(v, dtype), lse=lse, num_splits=splits)
    ref, ref_lse = oracle.attention_gqa(f64(q, dtype), f64(k, dtype), f64(v, dtype))
    check(o, ref, dtype, f"decode splits={splits}")
    assert_f32_close(lse.cpu().numpy(), ref_lse, atol=1e-3, what="lse")


def test_decode_full_size(osf):
    """The decode workload at full size: B=8, Hq=32, Hkv=8, Sk=32768, D=128, bf16 KV cache,
    every output element against the oracle."""
    B, Hq, Hkv, Sk, D = 8, 32, 8, 32768, 128
    q, k, v = si.qkv((B, Hq, 1, D), (B, Hkv, Sk, D), seed=0, dtype="bf16")
    o = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=True)
    ref, _ = oracle.attention_gqa(si.bf16_bits_to_f32(q), si.bf16_bits_to_f32(k), si.bf16_bits_to_f32(v))
    check(o, ref, "bf16", "decode full size")


@pytest.mark.parametrize("D", [64, 96, 128])
def test_decode_odd_shapes(osf, D):
    for (B, Hq, Hkv, Sk) in [(1, 4, 1, 1), (1, 4, 1, 63), (3, 6, 2, 1000), (1, 32, 8, 129)]:
        q, k, v = si.qkv((B, Hq, 1, D), (B, Hkv, Sk, D), seed=Sk + D, dtype="bf16")
        o = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v))
        ref, _ = oracle.attention_gqa(*(si.bf16_bits_to_f32(a) for a in (q, k, v)))
        check(o, ref, "bf16", f"decode {B},{Hq},{Hkv},{Sk},{D}")


# ----------------------------------------------------------------------- edge cases
def test_empty_problems_touch_nothing(osf):
    o = torch.full((1, 2, 0, 64), 7.0, device="cuda")
    q = torch.zeros(1, 2, 0, 64, device="cuda")
    k = torch.zeros(1, 2, 5, 64, device="cuda")
    osf.osf_attn_fwd_gqa(q, k, k, out=o)
    o = torch.full((1, 2, 3, 64), 7.0, device="cuda")
    q = torch.zeros(1, 2, 3, 64, device="cuda")
    k = torch.zeros(1, 2, 0, 64, device="cuda")
    osf.osf_attn_fwd_gqa(q, k, k, out=o)
    torch.cuda.synchronize()
    assert torch.all(o == 7.0)


def test_misaligned_views_still_correct(osf):
    # tensors starting one element past an allocation boundary: the kernels may not assume
    # 16-byte alignment
    B, Hq, Hkv, S, D = 1, 2, 1, 77, 64
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=9, dtype="bf16")
    def shifted(bits):
        t = torch.empty(bits.size + 1, dtype=torch.bfloat16, device="cuda")
        t[1:] = bf16_tensor(bits).reshape(-1)
        return t[1:].view(bits.shape)
    out = torch.empty(B * Hq * S * D + 1, dtype=torch.bfloat16, device="cuda")[1:].view(B, Hq, S, D)
    osf.osf_attn_fwd_gqa(shifted(q), shifted(k), shifted(v), out=out, causal=True)
    ref, _ = oracle.attention_gqa(*(si.bf16_bits_to_f32(a) for a in (q, k, v)), causal=True)
    check(out, ref, "bf16", "misaligned")


def test_output_guard_bands_untouched(osf):
    B, Hq, Hkv, S, D = 1, 4, 2, 300, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=10, dtype="bf16")
    n = B * Hq * S * D
    guard = 4096
    buf = torch.full((n + 2 * guard,), -12345.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(B, Hq, S, D)
    lse_buf = torch.full((B * Hq * S + 2 * guard,), -777.0, device="cuda")
    lse = lse_buf[guard:guard + B * Hq * S].view(B, Hq, S)
    osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), out=out, causal=True, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == -12345.0) and torch.all(buf[guard + n:] == -12345.0)
    assert torch.all(lse_buf[:guard] == -777.0) and torch.all(lse_buf[guard + B * Hq * S:] == -777.0)
    ref, _ = oracle.attention_gqa(*(si.bf16_bits_to_f32(a) for a in (q, k, v)), causal=True)
    check(out, ref, "bf16", "guard bands")


def test_invalid_arguments_on_device(osf):
    q = torch.zeros(1, 3, 8, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 8, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(osf.OsfError) as e:
        osf.osf_attn_fwd_gqa(q, k, k)
    assert e.value.status == osf.OSF_ERR_INVALID
    q = torch.zeros(1, 2, 8, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 9, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(osf.OsfError):
        osf.osf_attn_fwd_gqa(q, k, k, causal=True)
    with pytest.raises(osf.OsfError):
        osf.osf_attn_fwd_gqa(q, k, k, out=q)           # output aliases an input
    assert osf.osf_device_status() == osf.OSF_OK


def test_extreme_scores_stay_finite(osf):
    # large-magnitude scores: the running max must keep every exponent <= 0
    B, Hq, Hkv, S, D = 1, 2, 1, 200, 64
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=12)
    q = q * 30.0
    for dtype in ("f32", "bf16"):
        qq, kk, vv = (si.f32_to_bf16_bits(a) for a in (q, k, v)) if dtype == "bf16" else (q, k, v)
        o = osf.osf_attn_fwd_gqa(dev(qq, dtype), dev(kk, dtype), dev(vv, dtype), causal=True)
        ref, _ = oracle.attention_gqa(f64(qq, dtype), f64(kk, dtype), f64(vv, dtype), causal=True)
        check(o, ref, dtype, f"extreme {dtype}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_on_every_key_tile(osf, D, causal):
    """Keys scaled up along the sequence (key s by 1 + s/64), so a row's maximum grows by more
    than the lazy-rescale threshold on almost every key tile: O is rescaled between P V
    products on persistent multi-item CTAs (320 items, 8 key tiles each), where at D = 64 a
    tile's earlier P V may still be queued behind later score products."""
    B, Hq, Hkv, S = 2, 40, 8, 1024
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=D + causal)
    k = (k * (1.0 + np.arange(S, dtype=np.float32) / 64.0)[None, None, :, None]).astype(np.float32)
    qq, kk, vv = (si.f32_to_bf16_bits(a) for a in (q, k, v))
    o = osf.osf_attn_fwd_gqa(dev(qq, "bf16"), dev(kk, "bf16"), dev(vv, "bf16"), causal=causal)
    ref, _ = oracle.attention_gqa(f64(qq, "bf16"), f64(kk, "bf16"), f64(vv, "bf16"), causal=causal)
    check(o, ref, "bf16", f"rescale every tile D={D} causal={causal}")
    assert osf.osf_device_status() == osf.OSF_OK
