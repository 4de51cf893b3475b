"""The multi-kernel calls inside a captured CUDA graph: the float32 path (split pre-pass, forward,
combine), decode with its split combine, the chunked 1-D softmax and the tensor-core backward
(row-sum pre-pass, then the gradient grid) launch their later kernels as programmatic dependents of
the earlier ones.  A captured call must give exactly what the same call
gives eagerly (every kernel here is deterministic), after the outputs have been poisoned."""
import numpy as np
import pytest

import seeded_inputs as si
from conftest import bf16_tensor, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def eager_then_graph(fn, outs):
    """Run fn eagerly on a side stream, then capture it and replay; returns (eager, replayed)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    return eager, outs


def test_float32_tensor_core_path_in_a_graph(osf):
    B, H, S, D = 1, 2, 1024, 64
    q, k, v = (f32_tensor(a) for a in si.qkv((B, H, S, D), (B, H, S, D), seed=21))
    out = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda")
    ws = torch.empty(osf.osf_attn_workspace_bytes(osf.OSF_F32, B, H, H, S, S, D), dtype=torch.uint8, device="cuda")
    n0 = osf.osf_launch_count()
    eager, got = eager_then_graph(lambda: osf.osf_attn_fwd_gqa(q, k, v, out=out, lse=lse, workspace=ws), [out, lse])
    assert osf.osf_launch_count() - n0 >= 3   # pre-pass, forward, combine (counted again by the capture)
    for e, g_ in zip(eager, got):
        assert torch.equal(e, g_)


def test_decode_with_split_combine_in_a_graph(osf):
    B, Hq, Hkv, Sk, D = 2, 8, 2, 8192, 128
    q, k, v = (bf16_tensor(a) for a in si.qkv((B, Hq, 1, D), (B, Hkv, Sk, D), seed=22, dtype="bf16"))
    out = torch.empty_like(q)
    ws = torch.empty(osf.osf_attn_decode_workspace_bytes(osf.OSF_BF16, B, Hq, Hkv, Sk, D, 8), dtype=torch.uint8,
                     device="cuda")
    eager, got = eager_then_graph(lambda: osf.osf_attn_decode_gqa(q, k, v, out=out, num_splits=8, workspace=ws), [out])
    assert torch.equal(eager[0], got[0])


def test_chunked_softmax_in_a_graph(osf):
    x = f32_tensor(si.normal_f32((1, 1 << 22), 23, si.STREAM_X) * np.float32(8))
    z = torch.empty_like(x)
    ws = torch.empty(osf.osf_softmax_workspace_bytes(1, 1 << 22), dtype=torch.uint8, device="cuda")
    eager, got = eager_then_graph(lambda: osf.osf_softmax_rows(x, z, workspace=ws), [z])
    assert torch.equal(eager[0], got[0])


def test_tensor_core_backward_in_a_graph(osf):
    """The row-sum pre-pass, then the dK/dV grid (storing dS) as its dependent, then the dQ
    product over the stored dS as the dK/dV grid's dependent."""
    B, Hq, Hkv, S, D = 1, 4, 2, 640, 128
    q, k, v = (bf16_tensor(a) for a in si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=24, dtype="bf16"))
    g = bf16_tensor(si.qkv((B, Hq, S, D), (1, 1, 1, D), seed=25, dtype="bf16")[0])
    lse = torch.empty(B, Hq, S, device="cuda")
    o = osf.osf_attn_fwd_gqa_ex(q, k, v, mask="top_left", lse=lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(osf.osf_attn_bwd_workspace_bytes(osf.OSF_BF16, B, Hq, Hkv, S, S, D), dtype=torch.uint8,
                     device="cuda")
    n0 = osf.osf_launch_count()
    eager, got = eager_then_graph(
        lambda: osf.osf_attn_bwd_gqa(q, k, v, o, g, lse, dq=dq, dk=dk, dv=dv, mask="top_left", workspace=ws),
        [dq, dk, dv])
    # three launches, counted on the host for the eager run and for the capture
    assert osf.osf_launch_count() - n0 == 6
    for e, g_ in zip(eager, got):
        assert torch.equal(e, g_)
