"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics fix: the worked
rescale example of "softmax_attention" ("实现思路"), the N = 100 tail of the same section,
rows summing to one ("Softmax 算子的实现与优化", "Online Softmax" invariant), shift invariance
("Triton 版本 · Baseline"), the causal first row and GQA grouping of
"从零开始写Qwen3（五-其一）使用Triton实现自注意力" ("自注意力原理", "GQA"), brute force with
``math.fsum`` on tiny inputs, closed forms, and torch's fp64 CPU routines as a second witness.
A plausible slip in the oracle (a dropped scale, a wrong sign, a transposed operand, a wrong kv
head, an upper instead of lower triangle, a missing normalisation) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import read_golden


# ----------------------------------------------------------------------------- brute force
def brute_attention(Q, K, V, scale=None, causal=False):
    """Scalar loops with math.fsum / math.exp: no numpy arithmetic, no shared code."""
    M, d = len(Q), len(Q[0])
    N = len(K)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O, lse = [], []
    for i in range(M):
        s = []
        for j in range(N):
            if causal and j > i:
                continue
            s.append((j, math.fsum(Q[i][k] * K[j][k] for k in range(d)) * scale))
        mx = max(v for _, v in s)
        w = [(j, math.exp(v - mx)) for j, v in s]
        den = math.fsum(x for _, x in w)
        O.append([math.fsum(x * V[j][c] for j, x in w) / den for c in range(len(V[0]))])
        lse.append(mx + math.log(den))
    return np.array(O), np.array(lse)


def brute_softmax_row(x):
    mx = max(x)
    e = [math.exp(v - mx) for v in x]
    den = math.fsum(e)
    return [v / den for v in e]


def rnd(shape, seed, stream=si.STREAM_Q, scale=1.0):
    return si.normal_f32(shape, seed, stream, scale).astype(np.float64)


# ----------------------------------------------------------------------- worked example
def test_worked_rescale_example():
    g = read_golden("worked_rescale_example.txt")
    blocks = g["block"]
    x = [v for b in blocks for v in b]
    trace = []
    m, l = oracle.online_softmax_state(x, block=len(blocks[0]), trace=trace)
    # running maxima claimed by the page
    assert [t[0] for t in trace] == g["max_after"][0]
    # rescale factor exp(m_prev - m_new): exp(3 - 10) when the maximum jumps from 3 to 10
    assert trace[1][2] == pytest.approx(math.exp(g["alpha_exponent"][0][1]), rel=1e-15)
    # closed forms of the denominator under each reference maximum
    l1 = math.fsum(math.exp(v - 3.0) for v in blocks[0])
    assert trace[0][1] == pytest.approx(l1, rel=1e-15)
    l2 = math.fsum(math.exp(v - 10.0) for v in x)
    assert l == pytest.approx(l2, rel=1e-15)
    # old terms carried by alpha + new terms equals the direct sum (the page's point)
    carried = l1 * math.exp(3.0 - 10.0) + math.fsum(math.exp(v - 10.0) for v in blocks[1])
    assert carried == pytest.approx(l2, rel=1e-15)
    # the final softmax over all six scores
    z = oracle.softmax(np.array(x))
    assert np.allclose(z, [math.exp(v - 10.0) / l2 for v in x], rtol=1e-14, atol=0)
    # and the attention recurrence gives the same weights (V = identity picks them out)
    q = np.array([1.0])
    K = np.array(x)[:, None]
    V = np.eye(6)
    o, m_att, l_att = oracle.online_attention_row(q, K, V, block=3, scale=1.0)
    assert np.allclose(o, z, rtol=1e-14, atol=0)
    assert m_att == 10.0 and l_att == pytest.approx(l2, rel=1e-15)


# ---------------------------------------------------------------------------- tail mask
def test_tail_mask_n100():
    g = read_golden("tail_mask_n100.txt")
    M, N, d, blk = (int(g[k][0][0]) for k in ("M", "N", "d", "block"))
    first = int(g["last_block_first"][0][0])
    valid = int(g["last_block_valid"][0][0])
    nblk = -(-N // blk)
    assert (nblk - 1) * blk == first and N - first == valid
    Q = rnd((M, d), 11, si.STREAM_Q)
    K = rnd((N, d), 11, si.STREAM_K)
    V = rnd((N, d), 11, si.STREAM_V)
    O, lse = oracle.attention(Q, K, V)
    Ob, lseb = brute_attention(Q.tolist(), K.tolist(), V.tolist())
    assert np.max(np.abs(O - Ob)) < 1e-13
    assert np.max(np.abs(lse - lseb)) < 1e-12
    # the blocked recurrence over zero-padded keys with the -inf tail mask agrees ...
    Kp = np.vstack([K, np.zeros((nblk * blk - N, d))])
    Vp = np.vstack([V, np.zeros((nblk * blk - N, d))])
    for i in (0, 17, M - 1):
        o, _, _ = oracle.online_attention_row(Q[i], Kp, Vp, block=blk, n_keys=N)
        assert np.max(np.abs(o - O[i])) < 1e-13
    # ... and a planted mistake (padded keys kept, scored 0 instead of -inf) is detected.
    O_bad, _ = oracle.attention(Q, np.vstack([K, np.zeros((nblk * blk - N, d))]),
                                Vp)
    assert np.max(np.abs(O_bad - O)) > 1e-3


# ---------------------------------------------------------------------- sums and shifts
def test_softmax_rows_sum_to_one():
    x = si.softmax_rows_input(16, 1000, 5)
    z = oracle.softmax(x)
    sums = np.array([math.fsum(r) for r in z])
    assert np.max(np.abs(sums - 1.0)) < 1e-12
    assert np.all(z >= 0)


def test_attention_weights_sum_to_one():
    Q = rnd((37, 16), 3)
    K = rnd((53, 16), 3, si.STREAM_K)
    for causal in (False, True):
        O, _ = oracle.attention(Q, K, np.ones((53, 5)), causal=causal)
        assert np.max(np.abs(O - 1.0)) < 1e-13


@pytest.mark.parametrize("c", [-50.0, 7.5, 1e3])
def test_softmax_shift_invariance(c):
    x = rnd((8, 300), 4, si.STREAM_X, 8.0)
    z0 = oracle.softmax(x)
    z1 = oracle.softmax(x + c)
    assert np.all(np.isfinite(z1))
    assert np.max(np.abs(z1 - z0)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_attention_key_shift_invariance(causal):
    # adding one vector u to every key shifts all scores of row i by the same q_i . u * scale
    Q = rnd((29, 8), 6)
    K = rnd((29, 8), 6, si.STREAM_K)
    V = rnd((29, 8), 6, si.STREAM_V)
    u = 3.0 * rnd((8,), 7)
    O0, lse0 = oracle.attention(Q, K, V, causal=causal)
    O1, lse1 = oracle.attention(Q, K + u[None, :], V, causal=causal)
    assert np.max(np.abs(O1 - O0)) < 1e-12
    # lse shifts by exactly that common amount
    assert np.max(np.abs((lse1 - lse0) - (Q @ u) * 8 ** -0.5)) < 1e-12


# ----------------------------------------------------------------------- causal and GQA
def test_causal_row0_is_v0():
    B, Hq, Hkv, S, D = 2, 4, 2, 9, 8
    Q = rnd((B, Hq, S, D), 8)
    K = rnd((B, Hkv, S, D), 8, si.STREAM_K)
    V = rnd((B, Hkv, S, D), 8, si.STREAM_V)
    O, _ = oracle.attention_gqa(Q, K, V, causal=True)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(O[b, h, 0], V[b, h // (Hq // Hkv), 0])
    # row i sees keys 0..i only: changing key/value i+1.. leaves row i unchanged
    K2, V2 = K.copy(), V.copy()
    K2[:, :, 5:] += 1.0
    V2[:, :, 5:] -= 2.0
    O2, _ = oracle.attention_gqa(Q, K2, V2, causal=True)
    assert np.array_equal(O2[:, :, :5], O[:, :, :5])
    assert np.max(np.abs(O2[:, :, 5:] - O[:, :, 5:])) > 1e-3


def test_gqa_equals_mha_with_repeat_interleave():
    g = read_golden("gqa_head_geometry.txt")
    Hq, Hkv, D, G = (int(g[k][0][0]) for k in ("Hq", "Hkv", "D", "group"))
    assert Hq // Hkv == G
    B, Sq, Sk = 1, 5, 7
    Q = rnd((B, Hq, Sq, D), 9)
    K = rnd((B, Hkv, Sk, D), 9, si.STREAM_K)
    V = rnd((B, Hkv, Sk, D), 9, si.STREAM_V)
    O, lse = oracle.attention_gqa(Q, K, V)
    Om, lsem = oracle.attention_gqa(Q, np.repeat(K, G, axis=1), np.repeat(V, G, axis=1))
    assert np.max(np.abs(O - Om)) < 1e-13 and np.max(np.abs(lse - lsem)) < 1e-12
    # the other grouping (q head h -> kv head h % Hkv) is a different result
    Ow, _ = oracle.attention_gqa(Q, np.tile(K, (1, G, 1, 1)), np.tile(V, (1, G, 1, 1)))
    assert np.max(np.abs(Ow - O)) > 1e-2


def test_gqa_rejects_indivisible_heads():
    with pytest.raises(ValueError):
        oracle.attention_gqa(np.zeros((1, 3, 2, 4)), np.zeros((1, 2, 2, 4)), np.zeros((1, 2, 2, 4)))


def test_decode_row_sees_all_keys_even_if_causal():
    # seq_len_q == 1: the causal mask is not applied ("自注意力原理")
    Q = rnd((1, 4, 1, 8), 10)
    K = rnd((1, 2, 6, 8), 10, si.STREAM_K)
    V = rnd((1, 2, 6, 8), 10, si.STREAM_V)
    Oc, _ = oracle.attention_gqa(Q, K, V, causal=True)
    On, _ = oracle.attention_gqa(Q, K, V, causal=False)
    assert np.array_equal(Oc, On)


def test_attention_rows_matches_full():
    Q = rnd((2, 4, 33, 8), 12)
    K = rnd((2, 2, 33, 8), 12, si.STREAM_K)
    V = rnd((2, 2, 33, 8), 12, si.STREAM_V)
    for causal in (False, True):
        O, lse = oracle.attention_gqa(Q, K, V, causal=causal)
        rows = [(0, 0, 0), (1, 3, 32), (0, 2, 17), (1, 1, 5)]
        o, l = oracle.attention_rows(Q, K, V, rows, causal=causal)
        for n, (b, h, i) in enumerate(rows):
            assert np.max(np.abs(o[n] - O[b, h, i])) < 1e-14
            assert abs(l[n] - lse[b, h, i]) < 1e-13


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("M,N,d,causal", [(1, 1, 1, False), (3, 5, 2, False), (8, 8, 4, True),
                                          (6, 8, 3, True), (8, 7, 4, False), (5, 2, 4, False)])
def test_brute_force_tiny(M, N, d, causal):
    Q = rnd((M, d), 13) * 2
    K = rnd((N, d), 13, si.STREAM_K) * 2
    V = rnd((N, d), 13, si.STREAM_V)
    if causal and N < M:
        pytest.skip("causal needs N >= M for every row to have a key here")
    O, lse = oracle.attention(Q, K, V, causal=causal)
    Ob, lseb = brute_attention(Q.tolist(), K.tolist(), V.tolist(), causal=causal)
    assert np.max(np.abs(O - Ob)) < 1e-14
    assert np.max(np.abs(lse - lseb)) < 1e-13


def test_brute_force_explicit_scale():
    Q, K, V = rnd((4, 3), 14), rnd((6, 3), 14, si.STREAM_K), rnd((6, 2), 14, si.STREAM_V)
    O, _ = oracle.attention(Q, K, V, scale=0.37)
    Ob, _ = brute_attention(Q.tolist(), K.tolist(), V.tolist(), scale=0.37)
    assert np.max(np.abs(O - Ob)) < 1e-14


def test_softmax_spec_shape_brute_force():
    g = read_golden("softmax_spec_shape.txt")
    rows, T = int(g["rows"][0][0]), int(g["T"][0][0])
    x = si.softmax_rows_input(rows, T, 15)
    z = oracle.softmax(x)
    for r in range(rows):
        assert np.max(np.abs(z[r] - brute_softmax_row(x[r].astype(np.float64).tolist()))) < 1e-15


def test_scalar_flash_attention_d1():
    # "Puzzle 9: Simple FlashAttention": scalar q, k, v (d = 1, so d**-0.5 = 1);
    # z_i = sum_j softmax_j(q_i k_1..k_T) v_j.
    q, k, v = rnd((12,), 16), rnd((40,), 16, si.STREAM_K), rnd((40,), 16, si.STREAM_V)
    O, _ = oracle.attention(q[:, None], k[:, None], v[:, None])
    for i in range(12):
        w = brute_softmax_row([q[i] * kj for kj in k])
        assert abs(O[i, 0] - math.fsum(a * b for a, b in zip(w, v))) < 1e-14


# ---------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_values(causal):
    V = rnd((10, 6), 17, si.STREAM_V)
    O, lse = oracle.attention(np.zeros((10, 4)), rnd((10, 4), 17, si.STREAM_K), V, causal=causal)
    for i in range(10):
        n = i + 1 if causal else 10
        assert np.max(np.abs(O[i] - V[:n].mean(axis=0))) < 1e-14
        assert abs(lse[i] - math.log(n)) < 1e-14


def test_single_key_returns_v0():
    V = rnd((1, 7), 18, si.STREAM_V)
    O, lse = oracle.attention(rnd((5, 7), 18), rnd((1, 7), 18, si.STREAM_K), V)
    assert np.array_equal(O, np.repeat(V, 5, axis=0))


@pytest.mark.parametrize("val", [0.0, 3.25, -200.0])
def test_constant_row_is_uniform(val):
    z = oracle.softmax(np.full((3, 257), val))
    assert np.max(np.abs(z - 1.0 / 257)) < 1e-17
    # the recurrence keeps m = -inf only before the first block (an initial m = 0 would
    # underflow an all -200 row to l = 0)
    m, l = oracle.online_softmax_state(np.full(257, val), 32)
    assert m == val and l == pytest.approx(257.0, rel=1e-15)


def test_spike_closed_form():
    T = 1000
    x = np.zeros(T)
    x[123] = 30.0
    z = oracle.softmax(x)
    assert z[123] == pytest.approx(math.exp(30) / (math.exp(30) + T - 1), rel=1e-15)
    assert z[0] == pytest.approx(1.0 / (math.exp(30) + T - 1), rel=1e-15)


# ------------------------------------------------------------- recurrence vs definition
@pytest.mark.parametrize("block", [1, 32, 128, 1000])
def test_online_softmax_block_invariance(block):
    x = si.softmax_rows_input(1, 1000, 19)[0].astype(np.float64)
    m, l = oracle.online_softmax_state(x, block)
    assert m == np.max(x)
    assert l == pytest.approx(math.fsum(math.exp(v - m) for v in x), rel=1e-13)
    assert np.max(np.abs(oracle.online_softmax(x, block) - oracle.softmax(x))) < 1e-15


@pytest.mark.parametrize("block", [1, 32, 128, 300])
def test_online_attention_row_block_invariance(block):
    Q, K, V = rnd((4, 16), 20), rnd((300, 16), 20, si.STREAM_K), rnd((300, 16), 20, si.STREAM_V)
    O, _ = oracle.attention(Q, K, V)
    for i in range(4):
        o, m, l = oracle.online_attention_row(Q[i], K, V, block)
        assert np.max(np.abs(o - O[i])) < 1e-13


@pytest.mark.parametrize("splits", [1, 2, 7, 16])
def test_split_combine_invariance(splits):
    Q, K, V = rnd((3, 32), 21), rnd((1000, 32), 21, si.STREAM_K), rnd((1000, 32), 21, si.STREAM_V)
    O, lse = oracle.attention(Q, K, V)
    bounds = np.linspace(0, 1000, splits + 1).astype(int)
    for i in range(3):
        ms, ls, accs = [], [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            o, m, l = oracle.online_attention_row(Q[i], K[a:b], V[a:b], block=64)
            ms.append(m)
            ls.append(l)
            accs.append(o * l)
        ms.append(-np.inf)   # an empty chunk contributes nothing
        ls.append(0.0)
        accs.append(np.zeros(32))
        o, l = oracle.combine_partials(ms, ls, accs)
        assert np.max(np.abs(o - O[i])) < 1e-13
        assert abs(l - lse[i]) < 1e-12


# ------------------------------------------------------------------------ library witness
def test_torch_fp64_witness_attention():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, Hq, Hkv, Sq, Sk, D = 2, 8, 2, 40, 40, 32
    Q = rnd((B, Hq, Sq, D), 22)
    K = rnd((B, Hkv, Sk, D), 22, si.STREAM_K)
    V = rnd((B, Hkv, Sk, D), 22, si.STREAM_V)
    for causal in (False, True):
        O, _ = oracle.attention_gqa(Q, K, V, causal=causal)
        G = Hq // Hkv
        Ot = F.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K).repeat_interleave(G, 1),
            torch.from_numpy(V).repeat_interleave(G, 1), is_causal=causal).numpy()
        assert np.max(np.abs(O - Ot)) < 1e-12


def test_torch_fp64_witness_softmax():
    torch = pytest.importorskip("torch")
    x = si.softmax_rows_input(8, 4096, 23).astype(np.float64)
    assert np.max(np.abs(oracle.softmax(x) - torch.softmax(torch.from_numpy(x), -1).numpy())) < 1e-14


def test_lse_matches_scipy_logsumexp():
    sp = pytest.importorskip("scipy.special")
    Q, K, V = rnd((9, 16), 24), rnd((50, 16), 24, si.STREAM_K), rnd((50, 16), 24, si.STREAM_V)
    _, lse = oracle.attention(Q, K, V, causal=True)
    S = Q @ K.T * 0.25
    for i in range(9):
        assert abs(lse[i] - sp.logsumexp(S[i, :i + 1])) < 1e-13


# ------------------------------------------------------------- mask alignment when Sq != Sk
@pytest.mark.parametrize("Sq,Sk", [(5, 5), (3, 11), (7, 4), (1, 9)])
def test_masked_rows_equal_unmasked_attention_on_the_key_prefix(Sq, Sk):
    """Each masked row is plain (unmasked) attention over the keys it may see: keys 0..i for
    top-left ([Q3] "自注意力原理", tril(ones(Sq, Sk))), 0..i + Sk - Sq for bottom-right."""
    rng = np.random.default_rng(Sq * 31 + Sk)
    B, Hq, Hkv, D = 1, 4, 2, 8
    Q = rng.standard_normal((B, Hq, Sq, D))
    K = rng.standard_normal((B, Hkv, Sk, D))
    V = rng.standard_normal((B, Hkv, Sk, D))
    for mask, off in (("top_left", 0), ("bottom_right", Sk - Sq)):
        O, lse = oracle.attention_gqa(Q, K, V, mask=mask)
        for hq in range(Hq):
            kvh = hq // (Hq // Hkv)
            for i in range(Sq):
                last = Sk - 1 if (mask == "top_left" and Sq == 1) else min(i + off, Sk - 1)
                if last < 0:
                    assert np.all(O[0, hq, i] == 0) and lse[0, hq, i] == -np.inf
                    continue
                o, l = oracle.attention(Q[0, hq, i:i + 1], K[0, kvh, :last + 1], V[0, kvh, :last + 1])
                np.testing.assert_allclose(O[0, hq, i], o[0], rtol=1e-13, atol=1e-13)
                assert abs(lse[0, hq, i] - l[0]) < 1e-12


def test_bottom_right_equals_top_left_when_square_and_no_mask_for_one_row():
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((2, 2, 6, 4)); K = rng.standard_normal((2, 1, 6, 4)); V = rng.standard_normal((2, 1, 6, 4))
    a = oracle.attention_gqa(Q, K, V, mask="bottom_right")
    b = oracle.attention_gqa(Q, K, V, causal=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    q1 = Q[:, :, :1]
    c = oracle.attention_gqa(q1, K, V, mask="bottom_right")
    d = oracle.attention_gqa(q1, K, V, mask="none")
    assert np.array_equal(c[0], d[0])


def test_bottom_right_brute_force_loops():
    """Bottom-right alignment by explicit loops (exp of each kept score over their sum)."""
    rng = np.random.default_rng(8)
    Sq, Sk, D = 3, 5, 2
    Q = rng.standard_normal((1, 1, Sq, D)); K = rng.standard_normal((1, 1, Sk, D)); V = rng.standard_normal((1, 1, Sk, D))
    O, lse = oracle.attention_gqa(Q, K, V, mask="bottom_right")
    for i in range(Sq):
        keep = [j for j in range(Sk) if j <= i + Sk - Sq]
        sc = [sum(Q[0, 0, i, t] * K[0, 0, j, t] for t in range(D)) / math.sqrt(D) for j in keep]
        mx = max(sc)
        w = [math.exp(x - mx) for x in sc]
        for c in range(D):
            ref = sum(wj * V[0, 0, j, c] for wj, j in zip(w, keep)) / sum(w)
            assert abs(O[0, 0, i, c] - ref) < 1e-13
        assert abs(lse[0, 0, i] - (mx + math.log(sum(w)))) < 1e-13


def test_attention_rows_follows_the_mask():
    rng = np.random.default_rng(9)
    Q = rng.standard_normal((1, 2, 4, 8)); K = rng.standard_normal((1, 1, 9, 8)); V = rng.standard_normal((1, 1, 9, 8))
    full, full_lse = oracle.attention_gqa(Q, K, V, mask="bottom_right")
    rows = [(0, h, i) for h in range(2) for i in range(4)]
    o, l = oracle.attention_rows(Q, K, V, rows, mask="bottom_right")
    np.testing.assert_allclose(o, np.stack([full[0, h, i] for _, h, i in rows]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l, np.array([full_lse[0, h, i] for _, h, i in rows]), rtol=1e-13)


# --------------------------------------------------------------- scaled / causal row softmax
def test_softmax_masked_rows_equal_softmax_of_their_prefix():
    """Each row of the causal softmax is the plain softmax of the columns it keeps (0..r % P),
    zeros after; the scale multiplies before the max ([Q3] "使用triton实现")."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 7)) * 4
    for P, scale in ((10, 0.37), (4, 1.0), (0, 2.5)):
        z = oracle.softmax_masked(x, scale, P)
        for r in range(10):
            keep = 7 if P == 0 else min(7, r % P + 1)
            np.testing.assert_allclose(z[r, :keep], oracle.softmax(scale * x[r, :keep]), rtol=1e-14, atol=0)
            assert np.all(z[r, keep:] == 0)


def test_softmax_masked_defaults_are_the_plain_softmax():
    x = np.random.default_rng(4).standard_normal((5, 33))
    assert np.array_equal(oracle.softmax_masked(x), oracle.softmax(x))


def test_softmax_masked_brute_force():
    x = [[0.5, -1.0, 2.0, 0.25], [3.0, 1.0, -2.0, 0.0], [-1.0, -1.0, 4.0, 2.0]]
    z = oracle.softmax_masked(x, 0.5, 3)
    for r in range(3):
        keep = [0.5 * x[r][j] for j in range(4) if j <= r]
        mx = max(keep)
        den = sum(math.exp(v - mx) for v in keep)
        for j in range(4):
            ref = math.exp(0.5 * x[r][j] - mx) / den if j <= r else 0.0
            assert abs(z[r][j] - ref) < 1e-15


# ------------------------------------------------------------------- backward (gradients)
def _loss(Q, K, V, dO, mask):
    O, _ = oracle.attention_gqa(Q, K, V, mask=mask)
    return float(np.sum(O * dO))


@pytest.mark.parametrize("mask", ["none", "top_left", "bottom_right"])
def test_backward_matches_central_differences(mask):
    """dQ, dK, dV are the derivatives of L = sum(dO * O) through the forward definition:
    central differences of the forward oracle, element by element, on a small GQA case."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 3, 5, 3
    Q = rng.standard_normal((B, Hq, Sq, D)); K = rng.standard_normal((B, Hkv, Sk, D))
    V = rng.standard_normal((B, Hkv, Sk, D)); dO = rng.standard_normal((B, Hq, Sq, D))
    grads = oracle.attention_gqa_bwd(Q, K, V, dO, mask=mask)
    h = 1e-6
    for t, g in zip((Q, K, V), grads):
        num = np.zeros_like(t)
        for idx in np.ndindex(t.shape):
            keep = t[idx]
            t[idx] = keep + h; lp = _loss(Q, K, V, dO, mask)
            t[idx] = keep - h; lm = _loss(Q, K, V, dO, mask)
            t[idx] = keep
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_backward_single_key_closed_form():
    """One key: P = 1 whatever Q and K are, so O = V_0, dV_0 = sum_i dO_i, dQ = dK = 0."""
    rng = np.random.default_rng(12)
    Q = rng.standard_normal((1, 2, 4, 3)); K = rng.standard_normal((1, 1, 1, 3))
    V = rng.standard_normal((1, 1, 1, 3)); dO = rng.standard_normal((1, 2, 4, 3))
    dQ, dK, dV = oracle.attention_gqa_bwd(Q, K, V, dO)
    assert np.all(dQ == 0) and np.all(dK == 0)
    np.testing.assert_allclose(dV[0, 0, 0], dO[0].sum(axis=(0, 1)), rtol=1e-14)


def test_backward_uniform_attention_closed_form():
    """Q = 0: every row attends uniformly (P = 1/N).  Then dV_j = sum_i dO_i / N, dK = 0, and
    dQ_i = scale * sum_j (1/N)(dO_i.V_j - mean_k dO_i.V_k) K_j."""
    rng = np.random.default_rng(13)
    M, N, d = 3, 5, 4
    K = rng.standard_normal((N, d)); V = rng.standard_normal((N, d)); dO = rng.standard_normal((M, d))
    dQ, dK, dV = oracle.attention_bwd(np.zeros((M, d)), K, V, dO)
    s = d ** -0.5
    assert np.allclose(dK, 0, atol=0)
    for j in range(N):
        np.testing.assert_allclose(dV[j], dO.sum(axis=0) / N, rtol=1e-14)
    for i in range(M):
        a = np.array([dO[i] @ V[j] for j in range(N)])
        ref = s * sum((a[j] - a.mean()) / N * K[j] for j in range(N))
        np.testing.assert_allclose(dQ[i], ref, rtol=1e-13, atol=1e-15)


def test_backward_gqa_sums_the_heads_of_a_group():
    """A kv head's dK, dV are the sums of what each of its query heads sends back."""
    rng = np.random.default_rng(14)
    Q = rng.standard_normal((2, 4, 5, 3)); K = rng.standard_normal((2, 2, 6, 3))
    V = rng.standard_normal((2, 2, 6, 3)); dO = rng.standard_normal((2, 4, 5, 3))
    dQ, dK, dV = oracle.attention_gqa_bwd(Q, K, V, dO, mask="top_left")
    for b in range(2):
        for kvh in range(2):
            sk = np.zeros((6, 3)); sv = np.zeros((6, 3))
            for hq in (2 * kvh, 2 * kvh + 1):
                q, k, v = oracle.attention_bwd(Q[b, hq], K[b, kvh], V[b, kvh], dO[b, hq], q_index=np.arange(5))
                np.testing.assert_allclose(dQ[b, hq], q, rtol=1e-14)
                sk += k; sv += v
            np.testing.assert_allclose(dK[b, kvh], sk, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(dV[b, kvh], sv, rtol=1e-13, atol=1e-15)
