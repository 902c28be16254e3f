"""Naive (materialised) GPU attention -- the comparison baseline of the IO-aware path: a GEMM
writes S to HBM, this library's row-softmax kernel (C ABI ``fa_naive_softmax``) writes P and the
log-sum-exp, a GEMM forms O = P V. Checked against the fp64 oracle on the same seeded bf16
inputs with the tolerances of the fused path; its memory is checked to grow with N^2."""
import math

import numpy as np
import pytest

import oracle
from parity_util import assert_close_lse, assert_close_o, default_scale, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import naive
    return naive, oracle.oracle()


def _run(naive, bits, causal, scale):
    import torch
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o, lse = naive.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("cfg", [(1, 1, 256, 64, 1001), (4, 16, 2048, 64, 1002)],
                         ids=["B1H1N256d64", "B4H16N2048d64"])
def test_naive_matches_oracle(env, cfg):
    from exact_io_aware_fa_gb300 import synthetic
    naive, orc = env
    B, H, N, d, seed = cfg
    bits = synthetic.attention_inputs(B, H, N, d, seed=seed)
    o, lse = _run(naive, bits, False, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, default_scale(d))
    assert_close_o(o, o_ref, f"naive {cfg}")
    assert_close_lse(lse, lse_ref, f"naive {cfg}")


@pytest.mark.parametrize("N", [1, 17, 300, 513])
def test_naive_causal_small(env, N):
    from exact_io_aware_fa_gb300 import synthetic
    naive, orc = env
    bits = synthetic.attention_inputs(1, 2, N, 128, seed=600 + N, qk_sigma=1.5)
    o, lse = _run(naive, bits, True, default_scale(128))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], True, default_scale(128))
    assert_close_o(o, o_ref, f"naive causal N={N}", small_case=True)
    assert_close_lse(lse, lse_ref, f"naive causal N={N}")


@pytest.mark.parametrize("N,causal", [(4096, True), (4500, False), (4500, True), (1030, True),
                                     (8200, False)],
                         ids=["4096-causal", "4500", "4500-causal", "1030-causal", "8200"])
def test_naive_long_rows(env, N, causal):
    """Each softmax kernel of the naive path: a block per row for 1024 < N <= 8192 with N a
    multiple of 4 (4096, and 4500 with a ragged last vector), the two-pass warp kernel for
    N = 1030 (not a multiple of 4) and N = 8200 (beyond 8192)."""
    from exact_io_aware_fa_gb300 import synthetic
    naive, orc = env
    bits = synthetic.attention_inputs(1, 1, N, 64, seed=700 + N + int(causal))
    o, lse = _run(naive, bits, causal, default_scale(64))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(64))
    assert_close_o(o, o_ref, f"naive N={N} causal={causal}")
    assert_close_lse(lse, lse_ref, f"naive N={N} causal={causal}")


def test_naive_worked_example(env):
    """Scores [0,1,2,-1] against values [2,4,1,3] give 1.8619 ("15. FlashAttention", section
    "Worked example"), computed the materialised way."""
    naive, orc = env
    d, N = 64, 4
    q = np.zeros((1, 1, N, d), np.float32)
    k = np.zeros((1, 1, N, d), np.float32)
    v = np.zeros((1, 1, N, d), np.float32)
    q[0, 0, 0, 0] = 1.0
    k[0, 0, :, 0] = [0, 1, 2, -1]
    v[0, 0, :, 0] = [2, 4, 1, 3]
    bits = {n: (a.view(np.uint32) >> 16).astype(np.uint16) for n, a in (("q", q), ("k", k), ("v", v))}
    o, lse = _run(naive, bits, False, 1.0)
    # every normalised weight is rounded to bf16 before the PV product here (up to 2^-8 of itself,
    # times values up to 4), so the O tolerance applies rather than the output rounding alone
    assert abs(o[0, 0, 0, 0] - 1.8619) <= 1e-2
    assert abs(lse[0, 0, 0] - math.log(math.exp(0) + math.exp(1) + math.exp(2) + math.exp(-1))) <= 1e-3
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, 1.0)
    assert_close_o(o, o_ref, "naive unit", small_case=True)
    assert_close_lse(lse, lse_ref, "naive unit")


def test_naive_peak_memory_grows_with_n_squared(env):
    """The materialised path holds the N x N score (fp32) and probability (bf16) matrices; the
    fused forward holds only its inputs and outputs."""
    import torch
    from exact_io_aware_fa_gb300 import api
    naive, _ = env
    B, H, N, d = 1, 4, 4096, 64
    q = torch.randn(B, H, N, d, device="cuda", dtype=torch.bfloat16)
    k, v = torch.randn_like(q), torch.randn_like(q)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    naive.forward(q, k, v)
    torch.cuda.synchronize()
    naive_peak = torch.cuda.max_memory_allocated() - base
    torch.cuda.reset_peak_memory_stats()
    api.forward(q, k, v)
    torch.cuda.synchronize()
    fused_peak = torch.cuda.max_memory_allocated() - base
    nn = B * H * N * N
    assert naive_peak >= nn * (4 + 2)  # S in fp32 and P in bf16 at least
    # the fused forward holds O, LSE and, when it splits the keys of this small launch, fp32
    # partials of O -- all linear in N
    assert fused_peak * 8 <= naive_peak, (fused_peak, naive_peak)
