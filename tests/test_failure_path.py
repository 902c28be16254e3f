"""The kernels' failure path, exercised without a fault: a bounded mbarrier wait that nothing
completes gives up after a short limit, records its code in the device error word (read and
cleared by fa_device_error) and returns, and the CUDA context keeps working."""
import pytest

import oracle
from parity_util import assert_close_lse, assert_close_o, default_scale, to_dev, to_f64


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api
    return api, oracle.oracle()


@pytest.mark.gpu
def test_expired_wait_is_reported_and_context_survives(env):
    import time
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    assert api.device_error() == 0
    t0 = time.perf_counter()
    api.selftest_wait_timeout(20000)           # 20 ms limit
    code = api.device_error()                   # synchronises, reads and clears the word
    elapsed = time.perf_counter() - t0
    assert code == 1, code                      # code 1: a wait for a load gave up
    assert elapsed >= 0.015, elapsed            # it really waited for the limit
    assert api.device_error() == 0              # cleared
    # the context still runs attention exactly
    bits = synthetic.attention_inputs(1, 2, 200, 64, seed=4)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o, lse = api.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], True, default_scale(64))
    assert_close_o(to_f64(o), o_ref, "after timeout")
    assert_close_lse(to_f64(lse), lse_ref, "after timeout")


def test_selftest_rejects_bad_limit():
    from exact_io_aware_fa_gb300 import api, build
    build.build()
    lib = api.library()
    assert lib.fa_selftest_wait_timeout(0, None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(2000000, None) == api.FA_ERR_INVALID_ARG
