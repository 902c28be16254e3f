"""The entry points inside CUDA graphs: a forward + backward step captured once and replayed on
new inputs copied into the captured buffers must give the eager calls' results (O, LSE, dK,
dV bit for bit; dQ up to the order of its fp32 partial sums). Capture includes the dependent
launches between the backward's kernels (programmatic graph edges) and, for the host-buffer
step, the copies and the library's internal streams joined back into the captured stream."""
import pytest

from parity_util import same_up_to_summation_order

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api as a
    return a


@pytest.mark.parametrize("causal,window,d", [(False, -1, 64), (True, -1, 128), (True, 300, 64)])
def test_forward_backward_replay(api, causal, window, d):
    import torch
    B, Hq, Hkv, T = 2, 8, 4, 700
    gen = torch.Generator(device="cuda").manual_seed(5)

    def inputs():
        q = torch.randn(B, Hq, T, d, device="cuda", generator=gen).bfloat16()
        k = torch.randn(B, Hkv, T, d, device="cuda", generator=gen).bfloat16()
        v = torch.randn(B, Hkv, T, d, device="cuda", generator=gen).bfloat16()
        do = torch.randn(B, Hq, T, d, device="cuda", generator=gen).bfloat16()
        return q, k, v, do

    sq, sk, sv, sdo = inputs()  # the captured (static) buffers
    o = torch.empty_like(sq)
    lse = torch.empty(B, Hq, T, device="cuda")
    dq, dk, dv = torch.empty_like(sq), torch.empty_like(sk), torch.empty_like(sv)
    ws = torch.empty(api.backward_workspace_bytes(B, Hq, T, d), dtype=torch.uint8, device="cuda")

    def step(stream=None):
        api.forward(sq, sk, sv, causal=causal, window=window, out=o, lse=lse, nsplit=1,
                    stream=stream)
        api.backward(sq, sk, sv, o, lse, sdo, causal=causal, window=window, dq=dq, dk=dk, dv=dv,
                     workspace=ws, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s.cuda_stream)  # warm-up outside capture (first-call lookups)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        q, k, v, do = inputs()
        sq.copy_(q), sk.copy_(k), sv.copy_(v), sdo.copy_(do)
        g.replay()
        torch.cuda.synchronize()
        assert api.device_error() == 0
        o2, l2 = api.forward(q, k, v, causal=causal, window=window, nsplit=1)
        g2 = api.backward(q, k, v, o2, l2, do, causal=causal, window=window)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, l2)
        assert torch.equal(dk, g2[1]) and torch.equal(dv, g2[2])
        assert same_up_to_summation_order(dq, g2[0])


def test_host_step_replay(api):
    import torch
    B, Hq, Hkv, T, d = 2, 4, 2, 300, 64
    mk = lambda *shape: torch.randn(*shape).bfloat16().pin_memory()
    hq, hk, hv, hdo = mk(B, Hq, T, d), mk(B, Hkv, T, d), mk(B, Hkv, T, d), mk(B, Hq, T, d)
    outs = (torch.empty(B, Hq, T, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hq, T).pin_memory(),
            torch.empty(B, Hq, T, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hkv, T, d, dtype=torch.bfloat16).pin_memory(),
            torch.empty(B, Hkv, T, d, dtype=torch.bfloat16).pin_memory())
    buf = torch.empty(api.host_step_device_bytes(B, Hq, Hkv, T, T, d, 2), dtype=torch.uint8,
                      device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        api.forward_backward_host(hq, hk, hv, hdo, causal=True, nchunks=2, out=outs,
                                  device_buffer=buf, stream=s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.forward_backward_host(hq, hk, hv, hdo, causal=True, nchunks=2, out=outs,
                                  device_buffer=buf,
                                  stream=torch.cuda.current_stream().cuda_stream)
    for seed in (1, 2):
        torch.manual_seed(seed)
        for t in (hq, hk, hv, hdo):
            t.copy_(torch.randn(t.shape).bfloat16())
        g.replay()
        torch.cuda.synchronize()
        ref = api.forward_backward_host(hq, hk, hv, hdo, causal=True, nchunks=2)
        torch.cuda.synchronize()
        assert api.device_error() == 0
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), outs, ref):
            if name == "dQ":
                assert same_up_to_summation_order(a, b), name
            else:
                assert torch.equal(a, b), name
