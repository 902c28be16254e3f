"""Backward parity: dQ, dK, dV from the CUDA path (fed with the CUDA forward's O and LSE,
as a training step would) against the fp64 oracle's gradients of sum(O * dO) on the same
seeded bf16 inputs. Small/ragged sizes in full; the full-size configurations in full
(B=4 H=16 N=2048 d=64) or on seeded query/key row samples (B=4 H=16 N=4096 d=128)."""
import numpy as np
import pytest

import oracle
from parity_util import assert_close_grad, default_scale, to_dev, to_f64

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


def run_fwd_bwd(api, bits, causal, scale, workspace=True):
    import torch
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=causal, scale=scale)
    B, H, N, d = q.shape
    if workspace:
        ws = torch.empty(api.backward_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
        dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=causal, scale=scale, workspace=ws)
    else:
        # raw call with workspace = NULL (the Python wrapper always passes a buffer)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        st = api.backward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                              int(causal), scale, 0, torch.cuda.current_stream().cuda_stream)
        assert st == api.FA_OK
    torch.cuda.synchronize()
    assert api.device_error() == 0
    return to_f64(dq), to_f64(dk), to_f64(dv)


def check_full(api, orc, bits, causal, scale, what, workspace=True):
    g = run_fwd_bwd(api, bits, causal, scale, workspace)
    ref = orc.backward_bf16(bits["q"], bits["k"], bits["v"], bits["do"], causal, scale)
    for name, a, b in zip(("dQ", "dK", "dV"), g, ref):
        assert_close_grad(a, b, name, what)


SMALL_N = [1, 17, 64, 127, 128, 129, 255, 300, 513]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_and_ragged_full(env, d, causal, N):
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(1, 2, N, d, seed=200 + N, with_dout=True)
    check_full(api, orc, bits, causal, default_scale(d), f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_library_allocated_workspace(env, d):
    """workspace = NULL: the library allocates and frees it on the stream."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(2, 2, 333, d, seed=77, with_dout=True)
    check_full(api, orc, bits, True, default_scale(d), f"ws=NULL d={d}", workspace=False)


def test_gradient_bounds_untouched(env):
    """Ragged N: nothing is written past the end of dQ, dK or dV."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    B, H, N, d = 1, 2, 200, 128
    bits = synthetic.attention_inputs(B, H, N, d, seed=3, with_dout=True)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=True)
    n_el = B * H * N * d
    bufs = [torch.full((n_el + 8192,), 5.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    views = [b[:n_el].view(B, H, N, d) for b in bufs]
    api.backward(q, k, v, o, lse, do, causal=True, dq=views[0], dk=views[1], dv=views[2])
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[n_el:] == 5.0)


def test_backward_full_b4_h16_n2048_d64(env):
    """B=4 H=16 N=2048 d=64, non-causal (the benchmark workload's backward), in full."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(4, 16, 2048, 64, seed=1002, with_dout=True)
    check_full(api, orc, bits, False, default_scale(64), "B4 H16 N2048 d64 backward")


def test_backward_full_b4_h16_n2048_d64_causal(env):
    """B=4 H=16 N=2048 d=64 under the causal mask, in full: every fold record and dQ accumulator
    row of 64 heads, with units of very unequal cost on the persistent grid."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(4, 16, 2048, 64, seed=1012, with_dout=True)
    check_full(api, orc, bits, True, default_scale(64), "B4 H16 N2048 d64 causal backward")


def test_backward_sampled_b4_h16_n4096_d128_causal(env):
    """B=4 H=16 N=4096 d=128, causal; dQ on seeded query rows, dK/dV on seeded key rows."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, H, N, d = 4, 16, 4096, 128
    bits = synthetic.attention_inputs(B, H, N, d, seed=1005, with_dout=True)
    dq, dk, dv = run_fwd_bwd(api, bits, True, default_scale(d))
    rq = synthetic.sample_rows(N, 32, 1005)
    rk = synthetic.sample_rows(N, 32, 2005)
    ref_q, ref_k, ref_v = orc.backward_rows_bf16(bits["q"], bits["k"], bits["v"], bits["do"], True,
                                                 default_scale(d), rq, rk)
    assert_close_grad(dq[:, :, rq], ref_q, "dQ", "B4 H16 N4096 d128 causal")
    assert_close_grad(dk[:, :, rk], ref_k, "dK", "B4 H16 N4096 d128 causal")
    assert_close_grad(dv[:, :, rk], ref_v, "dV", "B4 H16 N4096 d128 causal")
    for g in (dq, dk, dv):
        assert np.all(np.isfinite(g))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_persistent_many_units_per_cta(env, d, causal):
    """B*H*ceil(N/128) key tiles far above the SM count: every CTA of the persistent backward
    walks several units, carrying its barrier phases, Q/dO ring and dV/dK epilogues across
    them."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(2, 200, 300, d, seed=310 + d, with_dout=True)
    check_full(api, orc, bits, causal, default_scale(d), f"many units d={d} causal={causal}")


def test_causal_unit_order_in_several_head_chunks(env):
    """Causal launches order their units key tile by key tile inside chunks of KV heads whose
    Q, dO and fp32 dQ accumulator rows fit in 96 MB of L2, spread evenly over the chunks.
    B1 H42 N8192 d128 needs 8 MB per head: four chunks of 11, 11, 11 and 9 heads (the last one
    ragged). dQ on seeded query rows, dK/dV on seeded key rows."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, H, N, d = 1, 42, 8192, 128
    bits = synthetic.attention_inputs(B, H, N, d, seed=4040, with_dout=True)
    dq, dk, dv = run_fwd_bwd(api, bits, True, default_scale(d))
    rq = synthetic.sample_rows(N, 16, 4040)
    rk = synthetic.sample_rows(N, 16, 5040)
    ref_q, ref_k, ref_v = orc.backward_rows_bf16(bits["q"], bits["k"], bits["v"], bits["do"], True,
                                                 default_scale(d), rq, rk)
    assert_close_grad(dq[:, :, rq], ref_q, "dQ", "head chunks")
    assert_close_grad(dk[:, :, rk], ref_k, "dK", "head chunks")
    assert_close_grad(dv[:, :, rk], ref_v, "dV", "head chunks")


def test_long_sequence_sampled(env):
    """N = 32768 (causal, d=64, one head): 256 key-tile units of up to 256 query steps each;
    dQ on seeded query rows, dK/dV on seeded key rows against the oracle."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, H, N, d = 1, 1, 32768, 64
    bits = synthetic.attention_inputs(B, H, N, d, seed=4098, with_dout=True)
    dq, dk, dv = run_fwd_bwd(api, bits, True, default_scale(d))
    rq = synthetic.sample_rows(N, 16, 4098)
    rk = synthetic.sample_rows(N, 16, 5098)
    ref_q, ref_k, ref_v = orc.backward_rows_bf16(bits["q"], bits["k"], bits["v"], bits["do"], True,
                                                 default_scale(d), rq, rk)
    assert_close_grad(dq[:, :, rq], ref_q, "dQ", "N=32768")
    assert_close_grad(dk[:, :, rk], ref_k, "dK", "N=32768")
    assert_close_grad(dv[:, :, rk], ref_v, "dV", "N=32768")
