"""Seeded random shapes through the extended calls, forward (with and without key splits) and
backward, against the fp64 oracle: grouped heads, query offsets, windows, ragged lengths and both
head dimensions in combinations the hand-picked cases do not cover."""
import numpy as np
import pytest

import oracle
from parity_util import assert_close_grad, assert_close_lse, assert_close_o, default_scale, to_dev, to_f64

def _cases(n=64, seed=20261202):
    """(B, Hq, Hkv, Tq, Tk, d, causal, window, nsplit); nsplit 0 = the library's choice."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.integers(1, 3))
        Hkv = int(rng.integers(1, 4))
        group = int(rng.choice([1, 2, 4]))
        Hq = Hkv * group
        if B * Hq > 8:
            continue
        Tk = int(rng.integers(1, 600))
        causal = bool(rng.integers(0, 2))
        Tq = int(rng.choice([1, 2, 5, int(rng.integers(1, Tk + 1)), Tk]))
        Tq = min(Tq, Tk) if causal else Tq
        window = int(rng.integers(0, Tk + 40)) if causal and rng.integers(0, 2) else -1
        d = int(rng.choice([64, 128]))
        nsplit = int(rng.choice([0, 1, int(rng.integers(2, 9))]))
        out.append((B, Hq, Hkv, Tq, Tk, d, causal, window, nsplit))
    return out


CASES = _cases()


def ids(c):
    B, Hq, Hkv, Tq, Tk, d, causal, w, ns = c
    return f"B{B}Hq{Hq}Hkv{Hkv}Tq{Tq}Tk{Tk}d{d}{'c' if causal else 'n'}w{w}s{ns}"


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api
    return api, oracle.oracle()


def test_cases_are_valid():
    for B, Hq, Hkv, Tq, Tk, d, causal, window, nsplit in CASES:
        assert Hq % Hkv == 0 and 1 <= Tq and 1 <= Tk and (not causal or Tq <= Tk)
        assert window < 0 or causal


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=ids)
def test_random_shape(env, case):
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, causal, window, nsplit = case
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=11 * Tk + 3 * Tq + d,
                                         with_dout=True)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale, window=window,
                         nsplit=None if nsplit == 0 else nsplit)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], causal, scale, window)
    small = Tq * Tk < 4096 or 0 <= window < 16
    assert_close_o(to_f64(o), o_ref, ids(case), small_case=small)
    assert_close_lse(to_f64(lse), lse_ref, ids(case))
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref, sens = orc.backward_ex_sens(bits["q"], bits["k"], bits["v"], bits["do"], causal, scale,
                                     window)
    for name, a, b, s in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref, sens):
        assert_close_grad(to_f64(a), b, name, ids(case), sens=s)


def _medium_cases(n=8, seed=20261203):
    """(B, H, N, d, causal): multi-head shapes with many persistent units per CTA, ragged N and
    both unit orders of the causal launches."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.integers(1, 5))
        H = int(rng.integers(3, 41))
        if B * H > 48:
            continue
        N = int(rng.integers(700, 4097))
        out.append((B, H, N, int(rng.choice([64, 128])), bool(rng.integers(0, 2))))
    return out


MEDIUM = _medium_cases()


def mid_ids(c):
    B, H, N, d, causal = c
    return f"B{B}H{H}N{N}d{d}{'c' if causal else 'n'}"


@pytest.mark.gpu
@pytest.mark.parametrize("case", MEDIUM, ids=mid_ids)
def test_random_medium_shape_sampled(env, case):
    """Forward on seeded query rows; dQ on seeded query rows and dK, dV on seeded key rows."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, H, N, d, causal = case
    bits = synthetic.attention_inputs(B, H, N, d, seed=N + 13 * H + d, with_dout=True)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    rq = synthetic.sample_rows(N, 16, N + 1)
    rk = synthetic.sample_rows(N, 16, N + 2)
    o_ref, lse_ref = orc.forward_rows_bf16(bits["q"], bits["k"], bits["v"], causal, scale, rq)
    what = mid_ids(case)
    assert_close_o(to_f64(o)[:, :, rq], o_ref, what)
    assert_close_lse(to_f64(lse)[:, :, rq], lse_ref, what)
    ref_q, ref_k, ref_v = orc.backward_rows_bf16(bits["q"], bits["k"], bits["v"], bits["do"], causal,
                                                 scale, rq, rk)
    assert_close_grad(to_f64(dq)[:, :, rq], ref_q, "dQ", what)
    assert_close_grad(to_f64(dk)[:, :, rk], ref_k, "dK", what)
    assert_close_grad(to_f64(dv)[:, :, rk], ref_v, "dV", what)
