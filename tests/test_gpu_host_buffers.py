"""GPU parity of ``osf_attn_fwd_gqa_host`` (attention on host buffers, copies overlapped in
chunks of whole (batch, kv head) units) against the fp64 oracle and against the device-buffer
entry point on the same inputs.

Cases cover an uneven split into chunks (9 units -> 5 chunks), one unit, the decode path
(Sq = 1), the float32 CUDA-core path, pageable host memory, a non-default stream and two calls
in a row on one device buffer.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from conftest import assert_bf16_close, assert_f32_close, bf16_tensor, f32_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def host(a, dtype, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) if dtype == "bf16" \
        else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.pin_memory() if pin else t.clone()


def f64(a, dtype):
    return si.bf16_bits_to_f32(a).astype(np.float64) if dtype == "bf16" else a.astype(np.float64)


def run_case(osf, B, Hq, Hkv, Sq, Sk, D, dtype, causal, seed, pin=True):
    q, k, v = si.qkv((B, Hq, Sq, D), (B, Hkv, Sk, D), seed=seed, dtype=dtype)
    out = osf.osf_attn_fwd_gqa_host(host(q, dtype, pin), host(k, dtype, pin), host(v, dtype, pin), causal=causal)
    torch.cuda.synchronize()
    ref, _ = oracle.attention_gqa(f64(q, dtype), f64(k, dtype), f64(v, dtype), causal=causal)
    got = out.float().numpy()
    what = f"host {dtype} {B},{Hq},{Hkv},{Sq},{Sk},{D} causal={causal} pinned={pin}"
    if dtype == "bf16":
        assert_bf16_close(got, ref, what)
        d = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=causal)
    else:
        assert_f32_close(got, ref, what=what)
        d = osf.osf_attn_fwd_gqa(f32_tensor(q), f32_tensor(k), f32_tensor(v), causal=causal)
    torch.cuda.synchronize()
    # same kernels on the same values; a chunk may pick another key split than the whole problem
    diff = float(np.max(np.abs(got - d.float().cpu().numpy())))
    assert diff <= (2e-2 if dtype == "bf16" else 1e-4), f"{what}: differs from the device entry point by {diff}"


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,dtype,causal", [
    (2, 8, 2, 300, 300, 128, "bf16", True),     # 4 units, one per chunk
    (3, 6, 3, 130, 130, 64, "bf16", False),     # 9 units -> 5 chunks of 2, 2, 2, 2, 1
    (1, 4, 1, 257, 257, 128, "bf16", True),     # a single unit
    (2, 32, 8, 1, 777, 128, "bf16", False),     # decode path, 16 units
    (2, 2, 2, 100, 100, 32, "f32", True),       # float32 CUDA-core path
])
def test_host_entry_point(osf, B, Hq, Hkv, Sq, Sk, D, dtype, causal):
    run_case(osf, B, Hq, Hkv, Sq, Sk, D, dtype, causal, seed=B * 100 + Hq + D)


def test_host_entry_point_pageable_memory(osf):
    run_case(osf, 2, 4, 2, 200, 200, 128, "bf16", True, seed=5, pin=False)


def test_host_entry_point_side_stream_and_reused_buffer(osf):
    """Two calls in a row on one device buffer, enqueued on a non-default stream."""
    B, Hq, Hkv, S, D = 2, 8, 4, 256, 128
    n = osf.osf_attn_host_buffer_bytes(osf.OSF_BF16, B, Hq, Hkv, S, S, D, True)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    outs, refs = [], []
    with torch.cuda.stream(side):
        for seed in (11, 12):
            q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=seed, dtype="bf16")
            outs.append(osf.osf_attn_fwd_gqa_host(host(q, "bf16"), host(k, "bf16"), host(v, "bf16"), causal=True,
                                                  device_buffer=buf))
            refs.append(oracle.attention_gqa(f64(q, "bf16"), f64(k, "bf16"), f64(v, "bf16"), causal=True)[0])
    side.synchronize()
    for i, (o, r) in enumerate(zip(outs, refs)):
        assert_bf16_close(o.float().numpy(), r, f"call {i}")


def test_host_entry_point_rejects_small_buffer(osf):
    q = torch.zeros(1, 4, 64, 64, dtype=torch.bfloat16).pin_memory()
    k = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16).pin_memory()
    n = osf.osf_attn_host_buffer_bytes(osf.OSF_BF16, 1, 4, 2, 64, 64, 64, False)
    small = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(osf.OsfError) as e:
        osf.osf_attn_fwd_gqa_host(q, k, k.clone().pin_memory(), device_buffer=small)
    assert e.value.status == osf.OSF_ERR_WORKSPACE


def test_host_entry_point_full_size_gqa_causal_prefill(osf):
    """The GQA causal prefill workload (B=2, Hq=32, Hkv=8, S=4096, D=128, bf16) from pinned host
    buffers, as the benchmark runs it: sampled rows of every head against the oracle, and the
    whole output against the device-buffer entry point."""
    B, Hq, Hkv, S, D = 2, 32, 8, 4096, 128
    q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=0, dtype="bf16")
    out = osf.osf_attn_fwd_gqa_host(host(q, "bf16"), host(k, "bf16"), host(v, "bf16"), causal=True)
    d = osf.osf_attn_fwd_gqa(bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), causal=True)
    torch.cuda.synchronize()
    of = out.float().numpy()
    diff = float(np.max(np.abs(of - d.float().cpu().numpy())))
    assert diff <= 2e-2, f"host path differs from the device entry point by {diff}"
    rng = np.random.default_rng(1)
    rows = [(b, h, i) for b in range(B) for h in range(Hq)
            for i in (0, 255, 256, S - 1, int(rng.integers(0, S)))]
    ref, _ = oracle.attention_rows(f64(q, "bf16"), f64(k, "bf16"), f64(v, "bf16"), rows, causal=True)
    assert_bf16_close(np.stack([of[b, h, i] for b, h, i in rows]), ref, "host path full size")


def test_host_entry_point_concurrent_threads(osf):
    """Calls from two host threads at once, each on its own stream and device buffer (the library
    serialises their enqueueing on the shared copy streams): both results match the oracle."""
    import threading
    B, Hq, Hkv, S, D = 1, 8, 2, 384, 128
    cases = []
    for seed in (21, 22):
        q, k, v = si.qkv((B, Hq, S, D), (B, Hkv, S, D), seed=seed, dtype="bf16")
        cases.append((host(q, "bf16"), host(k, "bf16"), host(v, "bf16"),
                      oracle.attention_gqa(f64(q, "bf16"), f64(k, "bf16"), f64(v, "bf16"), causal=True)[0]))
    outs = [None, None]
    errors = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(3):
                    outs[i] = osf.osf_attn_fwd_gqa_host(*cases[i][:3], causal=True)
            st.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert_bf16_close(outs[i].float().numpy(), cases[i][3], f"thread {i}")
