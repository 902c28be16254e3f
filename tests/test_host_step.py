"""fa_forward_backward_host: one forward + backward step on host tensors, the KV heads cut into
chunks whose copies overlap the other chunks' kernels. Its results must equal the device calls'
on the same inputs -- O, LSE, dK and dV bit for bit (every head's arithmetic is the same kernel
work), dQ up to the order of its fp32 partial sums -- and the fp64 oracle's within tolerance."""
import numpy as np
import pytest

import oracle
from parity_util import (assert_close_grad, assert_close_lse, assert_close_o, default_scale,
                         same_up_to_summation_order, to_dev, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api
    return api, oracle.oracle()


def host(bits, pin=True):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


# (B, Hq, Hkv, Tq, Tk, d, causal, window, nchunks)
CASES = [
    (2, 4, 2, 300, 500, 64, True, -1, 3),      # grouped heads, offset, chunks of 1, 1, 2 KV heads
    (1, 4, 4, 257, 257, 128, False, -1, 0),    # library's chunk count
    (1, 6, 2, 400, 400, 64, True, 100, 16),    # window; more chunks than KV heads
    (3, 2, 1, 130, 700, 128, True, -1, 1),     # one chunk
    (2, 8, 2, 40, 500, 64, True, -1, 3),       # Tq <= 64: each chunk's forward packs its heads
]


def ids(c):
    B, Hq, Hkv, Tq, Tk, d, causal, w, n = c
    return f"B{B}Hq{Hq}Hkv{Hkv}Tq{Tq}Tk{Tk}d{d}{'c' if causal else 'n'}w{w}n{n}"


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_host_step_matches_device_calls_and_oracle(env, case):
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, causal, window, nchunks = case
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=11 * Tq + Tk, with_dout=True)
    scale = default_scale(d)
    hq, hk, hv, hdo = (host(bits[n]) for n in ("q", "k", "v", "do"))
    o, lse, dq, dk, dv = api.forward_backward_host(hq, hk, hv, hdo, causal=causal, scale=scale,
                                                   window=window, nchunks=nchunks)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    # the device calls on the same inputs (no key-range split, as the step runs fa_forward_ex)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    o2, lse2 = api.forward(q, k, v, causal=causal, scale=scale, window=window, nsplit=1)
    dq2, dk2, dv2 = api.backward(q, k, v, o2, lse2, do, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert torch.equal(o, o2.cpu()) and torch.equal(lse, lse2.cpu())
    assert torch.equal(dk, dk2.cpu()) and torch.equal(dv, dv2.cpu())
    assert same_up_to_summation_order(dq, dq2.cpu())
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], causal, scale, window)
    assert_close_o(to_f64(o), o_ref, ids(case), small_case=Tq * Tk < 4096)
    assert_close_lse(to_f64(lse), lse_ref, ids(case))
    ref = orc.backward_ex(bits["q"], bits["k"], bits["v"], bits["do"], causal, scale, window)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_close_grad(to_f64(a), b, name, ids(case))


def test_host_step_pageable_memory_and_reuse(env):
    """Pageable host tensors give the same results; two steps through one device buffer and
    one set of outputs, the second on different inputs, each match a fresh step."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    B, Hq, Hkv, Tq, Tk, d = 1, 4, 2, 200, 300, 64
    outs = None
    buf = torch.empty(api.host_step_device_bytes(B, Hq, Hkv, Tq, Tk, d, 2), dtype=torch.uint8,
                      device="cuda")
    for seed in (1, 2):
        bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=seed, with_dout=True)
        pinned = [host(bits[n]) for n in ("q", "k", "v", "do")]
        pageable = [host(bits[n], pin=False) for n in ("q", "k", "v", "do")]
        outs = api.forward_backward_host(*pageable, causal=True, nchunks=2, out=outs,
                                         device_buffer=buf)
        torch.cuda.synchronize()
        fresh = api.forward_backward_host(*pinned, causal=True, nchunks=2)
        torch.cuda.synchronize()
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), outs, fresh):
            if name == "dQ":
                assert same_up_to_summation_order(a, b), name
            else:
                assert torch.equal(a, b), name
    assert api.device_error() == 0


def test_host_step_without_query_rows_zeroes_dk_dv(env):
    import torch
    api, _ = env
    B, Hq, Hkv, Tq, Tk, d = 1, 2, 2, 0, 300, 128
    q = torch.empty((B, Hq, Tq, d), dtype=torch.bfloat16).pin_memory()
    k = torch.randn((B, Hkv, Tk, d)).bfloat16().pin_memory()
    v = torch.randn((B, Hkv, Tk, d)).bfloat16().pin_memory()
    dk = torch.full((B, Hkv, Tk, d), 7.0, dtype=torch.bfloat16).pin_memory()
    dv = torch.full((B, Hkv, Tk, d), 7.0, dtype=torch.bfloat16).pin_memory()
    o, lse, dq = (torch.empty_like(q), torch.empty((B, Hq, Tq), dtype=torch.float32),
                  torch.empty_like(q))
    api.forward_backward_host(q, k, v, q, causal=False, out=(o, lse, dq, dk, dv))
    torch.cuda.synchronize()
    assert api.device_error() == 0
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0
